// Ragged paged attention for prefill chunks on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), head_dim 48, 64 or 128.
//
// One CTA = (listed request, KV head, pair of 128-row query tiles).  A row
// is a (token, query head) pair of the KV head's group: 128/g consecutive
// new tokens x g heads per tile (the vllm-lite README's grouped-query fold,
// so one K/V tile feeds all g heads).  Query i of a request with t new
// tokens and context L sits at position L - t + i and sees keys 0 .. that
// position ("31. Engine v2", "Attention over the pool").  Keys come in
// tiles of 128 = 8 paged blocks; each block's 16-row K and V slices of this
// KV head are copied by TMA straight from the pool through the block table
// (key j lives in block table[j / 16], row j % 16).
//
// Warp roles (384 threads):
//   warps 0, 2  TMA producers: warp 0 both Q tiles once, then K tiles, warp 2
//               V tiles, each into a 2-stage ring (a K stage is refilled once
//               both S MMAs that read it are done, a V stage once both PV
//               MMAs are done); a tile's 16 boxes go out from 16 lanes at once;
//   warps 3..11 combined write + attention calls: when this CTA is the only
//               one of its request and KV head (one pair of tiles, uncut),
//               they first write the request's new K/V rows of that head
//               into the pool and signal the producers, which wait for it
//               before the first key tile that holds a new row (plain
//               launches only; the other requests' rows, and a mixed
//               launch's, come from a scatter ahead of the launch);
//   warp 1      MMA issuer (one thread) and TMEM owner; per key tile it
//               issues PV_a(j-1), S_a(j), PV_b(j-1), S_b(j), so the tensor
//               core always has the other tile's work while a softmax runs;
//   warps 4..7  softmax of tile a, warps 8..11 softmax of tile b, one row per
//               thread (= TMEM lane): two passes over the S row in TMEM (row
//               max, then exp2 in the log2 domain), P written back as bf16
//               pairs over the first half of the S columns, where the PV MMA
//               reads it as its A operand.  The running max only moves (and O
//               is rescaled in TMEM) when it grows by more than 2^8.  A CTA
//               with a single tile splits each row between warps w and w + 4,
//               one per 64-column half of S (and of O): they swap half-row
//               maxima and sums through shared memory, and each writes its
//               half of P over its own first 32 columns ([0,32) and [64,96)),
//               and S alternates between two TMEM buffers (the unused S_b
//               columns), so the MMA of key tile j+1 overlaps tile j's softmax.
// TMEM: S_a [0,128), S_b [128,256), O_a [256,384), O_b [384,512).
//
// Key pieces: a pair may be cut into consecutive ranges of key tiles, one
// CTA each (the planner does so for heavy pairs that would start in a later
// wave, to even out the SMs' loads).  When its loop is done, such a CTA
// counts itself on the pair's counter.  Every piece but the last to count
// writes its rows' unscaled O and (running max, weight sum) as fp32
// partials and signals them on the counter's second word; the last one
// waits (bounded) for those signals and merges the partials into its own O,
// still in tensor memory, with the exact split-softmax identity, writes the
// bf16 output and returns both words to zero.
// Shared memory (128-byte swizzle): Q_a, Q_b, K and V tiles as [128][64]
// sub-tiles, K-major for Q and K, MN-major for V.  Head dims below 64 are
// padded to 64 columns: the TMA box is 64 columns wide and fills the
// columns past head_dim with zeros, which add nothing to Q K^T and give
// zero output columns in P V that are not stored.
#include <climits>
#include <mutex>

#include "common.cuh"
#include "decode_warp.cuh"
#include "sm100.cuh"

namespace pkv {

constexpr int kTcThreads = 384;
constexpr int kTcRows = 128;          // query rows per tile (MMA M)
constexpr int kTcKeys = 128;          // keys per tile (MMA N of S, K of PV)
constexpr int kSub = 16384;           // one [128][64] bf16 sub-tile

// Shared-memory layout for a padded head dim DP (64 or 128).
template <int DP>
struct TcCfg {
    static constexpr int kHalves = DP / 64;            // 64-column sub-tiles per row
    static constexpr int kTile = kHalves * kSub;        // [128][DP]
    static constexpr int kQOff = 0;                     // Q_a, Q_b
    static constexpr int kKOff = kQOff + 2 * kTile;     // 2 stages
    static constexpr int kVOff = kKOff + 2 * kTile;     // 2 stages
    static constexpr int kBarOff = kVOff + 2 * kTile;
    static constexpr int kXOff = kBarOff + 256;        // softmax pair exchange: max [2][2][128], sum [2][128]
    static constexpr int kSmem = 1024 + kXOff + 3 * 1024;
    // mixed batches, decode CTAs: a ring of kDecStages stages (a K and a V
    // slice each) per warp, then their barriers
    static constexpr int kDecStages = DP == 128 ? 2 : 4;
    static constexpr int kDecRing = kDecStages * WarpRing<DP>::kStage;
    static constexpr int kDecBarOff = (kTcThreads / 32) * kDecRing;
    static constexpr int kSmemDec = 1024 + kDecBarOff + (kTcThreads / 32) * kDecStages * 8;
    static constexpr int kSmemMix = kSmem > kSmemDec ? kSmem : kSmemDec;
    static_assert(kSmemMix <= 227 * 1024, "the decode rings must fit a CTA's shared memory");
    // ... over a quantized pool (head dim 128): rings of E4M3 codes, then
    // every warp's scale array, then the barriers
    static constexpr int kDecStagesF8 = 4;
    static constexpr int kDecRingF8 = kDecStagesF8 * WarpRingF8::kStage;
    static constexpr int kDecScaleOffF8 = (kTcThreads / 32) * kDecRingF8;
    static constexpr int kDecBarOffF8 = kDecScaleOffF8 + (kTcThreads / 32) * kDecStagesF8 * WarpRingF8::kScaleStage;
    static constexpr int kSmemDecF8 = 1024 + kDecBarOffF8 + (kTcThreads / 32) * kDecStagesF8 * 8;
    static constexpr int kSmemMixF8 = kSmem > kSmemDecF8 ? kSmem : kSmemDecF8;
    static_assert(kSmemMixF8 <= 227 * 1024, "the decode rings must fit a CTA's shared memory");
};

constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;  // move the running max only when it grows by more than this

enum TcBar {
    kBarQ = 0,
    kBarK0 = 1, kBarK1 = 2,
    kBarV0 = 3, kBarV1 = 4,
    kBarSA = 5, kBarSB = 6,           // S of tile a / b done (also frees a K stage)
    kBarPA = 7, kBarPB = 8,           // P of tile a / b written (4 warps each)
    kBarOA = 9, kBarOB = 10,          // PV of tile a / b done (also frees a V stage)
    kBarMmaDone = 11,
    kBarOFin = 12,                    // single tile: every PV done (one phase)
    kNumTcBars = 13,
    kBarW = 13                        // OWN launches only: the CTA's own new K/V rows are in the pool
};

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: the A operand (P) read from tensor memory.
__device__ __forceinline__ void tc_mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Pass 1 of the softmax: max of the raw scores of NC columns of this
// thread's S row (TMEM columns at ts, keys key0 ..); keys past qpos, and
// keys at or below qlo (outside a sliding window, WIN), are masked when MASK.
template <bool MASK, int NC, bool WIN>
__device__ __forceinline__ float tc_row_max(uint32_t ts, int key0, int qpos, int qlo)
{
    float m[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
    for (int c = 0; c < NC / 32; c++) {
        uint32_t v[32];
        tmem_ld32(ts + c * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 32; k += 2) {
            float s0 = __uint_as_float(v[k]), s1 = __uint_as_float(v[k + 1]);
            if (MASK) {
                const int k0 = key0 + c * 32 + k;
                if (k0 > qpos || (WIN && k0 <= qlo)) s0 = -INFINITY;
                if (k0 + 1 > qpos || (WIN && k0 + 1 <= qlo)) s1 = -INFINITY;
            }
            m[(k >> 1) & 3] = max3f(m[(k >> 1) & 3], s0, s1);
        }
    }
    return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
}

// Pass 2: P = 2^(s * sl2 - ms) for NC columns at ts, as bf16 pairs written
// over the first NC/2 of them (each 16-column chunk goes over columns
// already read); returns this row's sum of P over them.
template <bool MASK, int NC, bool WIN>
__device__ __forceinline__ float tc_row_exp(uint32_t ts, int key0, int qpos, int qlo, float sl2, float ms)
{
    const uint64_t scale2 = f2_pack(sl2, sl2), neg2 = f2_pack(-ms, -ms);
    uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int c = 0; c < NC / 16; c++) {
        uint32_t v[16];
        tmem_ld16(ts + c * 16, v);
        tmem_ld_wait();
        uint32_t pw[8];
#pragma unroll
        for (int k = 0; k < 8; k++) {
            float s0 = __uint_as_float(v[2 * k]), s1 = __uint_as_float(v[2 * k + 1]);
            if (MASK) {
                const int k0 = key0 + c * 16 + 2 * k;
                if (k0 > qpos || (WIN && k0 <= qlo)) s0 = -INFINITY;
                if (k0 + 1 > qpos || (WIN && k0 + 1 <= qlo)) s1 = -INFINITY;
            }
            float t0, t1;
            f2_unpack(f2_fma(f2_pack(s0, s1), scale2, neg2), t0, t1);
            const float p0 = fast_exp2(t0), p1 = fast_exp2(t1);
            acc[k & 3] = f2_add(acc[k & 3], f2_pack(p0, p1));
            pw[k] = pack_bf16x2(p0, p1);
        }
        tmem_st8(ts + c * 8, pw);
    }
    tmem_st_wait();
    float sum = 0.f;
#pragma unroll
    for (int q = 0; q < 4; q++) {
        float a, b;
        f2_unpack(acc[q], a, b);
        sum += a + b;
    }
    return sum;
}

// O columns [32 c0, 32 (c0 + nc)) of this thread's TMEM row *= alpha.
__device__ __forceinline__ void tc_rescale_cols(uint32_t to, int c0, int nc, float alpha)
{
#pragma unroll 1
    for (int c = c0; c < c0 + nc; c++) {
        uint32_t ov[32];
        tmem_ld32(to + c * 32, ov);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 32; k++) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
        tmem_st32(to + c * 32, ov);
    }
    tmem_st_wait();
}

// Store O columns [32 c0, 32 (c0 + nc)) of this thread's row (clipped to D)
// as bf16, scaled by inv: row `row` of the tile is token tok0 + row / g,
// query head kh * g + row % g.
template <int D>
__device__ __forceinline__ void tc_store_rows(const AttnParams &p, uint32_t to, int row, int nr, int tok0, int kh,
                                              int g, float inv, int c0, int nc)
{
    const size_t orow = row < nr ? ((size_t)(tok0 + row / g) * p.hq + kh * g + row % g) * D : 0;
#pragma unroll 1
    for (int c = c0; c < c0 + nc; c++) {
        if (c * 32 >= D) break;                                     // warp-uniform
        uint32_t v[32];
        tmem_ld32(to + c * 32, v);
        tmem_ld_wait();
        if (row < nr) {
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow + c * 32);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                if (c * 32 + q * 8 >= D) break;                     // padding columns are not stored
                uint32_t w4[4];
#pragma unroll
                for (int e = 0; e < 4; e++)
                    w4[e] = pack_bf16x2(__uint_as_float(v[q * 8 + 2 * e]) * inv,
                                        __uint_as_float(v[q * 8 + 2 * e + 1]) * inv);
                dst[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        }
    }
}

// Store O columns [32 c0, 32 (c0 + nc)) of this thread's row (clipped to D)
// unscaled as an fp32 partial row `prow`, and with write_ml its running max
// (exp2 domain) and weight sum.  valid false: read TMEM only (the load is
// warp-collective), store nothing.
template <int D>
__device__ __forceinline__ void tc_store_partial(const AttnParams &p, uint32_t to, size_t prow, bool valid, float m,
                                                 float l, int c0, int nc, bool write_ml)
{
#pragma unroll 1
    for (int c = c0; c < c0 + nc; c++) {
        if (c * 32 >= D) break;                                     // warp-uniform
        uint32_t v[32];
        tmem_ld32(to + c * 32, v);
        tmem_ld_wait();
        if (valid) {
            float4 *dst = reinterpret_cast<float4 *>(p.part_o + prow * D + c * 32);
#pragma unroll
            for (int q = 0; q < 8; q++) {
                if (c * 32 + q * 4 >= D) break;
                dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                     __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
        }
    }
    if (valid && write_ml) p.part_ml[prow] = make_float2(m, l);
}

// Wait until *word reaches `target` (acquire), for at most the pipeline
// wait limit; on time-out flag kDevErrTimeout and return false.  Used by the
// last piece of a pair for the other pieces' partials: those CTAs are past
// their loops when they count, and only store their rows before they
// signal, so the wait ends.
__device__ __forceinline__ bool wait_count(const uint32_t *word, uint32_t target, uint32_t *err)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t i = 0; i < kWaitLimitIters; i++) {
        uint32_t v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(word) : "memory");
        if (v >= target) return true;
        if ((i & 63u) == 63u && globaltimer_ns() - t0 > kWaitLimitNs) break;
        __nanosleep(64);
    }
    atomicOr(err, kDevErrTimeout);
    return false;
}

// The end of a key piece, run by the 256 softmax threads (named barrier 7):
// this thread's row rr (0..255: tile a, then tile b) holds O columns
// [32 c0, 32 (c0 + nc)) in TMEM at `to`, with running max m (exp2 domain)
// and weight sum l over this piece's keys; write_ml: this thread reports
// (m, l) of its row.  ok: this thread's waits succeeded (CTA-uniform here).
// Counting, partial store / signal, or wait and merge, as described above.
template <int D>
__device__ __forceinline__ void tc_piece_epilogue(const AttnParams &p, uint32_t *cnt, size_t slot0, int piece,
                                                  int pieces, uint32_t to, int rr, bool valid, float m, float l,
                                                  int c0, int nc, bool write_ml, bool ok, size_t orow,
                                                  uint32_t *s_flag)
{
    named_bar_sync(7, 256);                                     // every row of the CTA has left its loop
    if (threadIdx.x == 128) {
        const uint32_t old = atomicAdd(cnt, 1u);
        if (old >= (uint32_t)pieces) atomicOr(p.err, kDevErrCounter);   // counters were not zero-filled
        s_flag[0] = old + 1u == (uint32_t)pieces ? 1u : 0u;
    }
    named_bar_sync(7, 256);
    if (s_flag[0] == 0u) {
        // not the last: partials out, then signal them (also after a failed
        // wait, so that the last piece's wait ends)
        tc_store_partial<D>(p, to, (slot0 + piece) * 256 + rr, valid && ok, m, l, c0, nc, write_ml);
        named_bar_sync(7, 256);
        if (threadIdx.x == 128) {
            __threadfence();                                    // release the partials (cumulative over the barrier)
            atomicAdd(cnt + 1, 1u);
        }
        return;
    }
    if (threadIdx.x == 128) s_flag[1] = wait_count(cnt + 1, (uint32_t)pieces - 1u, p.err) ? 1u : 0u;
    named_bar_sync(7, 256);
    if (s_flag[1] != 0u) {
        // row weights: M over every piece, the denominator over every piece
        float M = m;
        for (int q = 0; q < pieces; q++)
            if (q != piece && valid) M = fmaxf(M, __ldcg(&p.part_ml[(slot0 + q) * 256 + rr]).x);
        const float Ms = M == -INFINITY ? 0.f : M;
        const float w0 = exp2f(m - Ms);                          // 2^-inf = 0
        float den = w0 * l;
        for (int q = 0; q < pieces; q++) {
            if (q == piece || !valid) continue;
            const float2 ml = __ldcg(&p.part_ml[(slot0 + q) * 256 + rr]);
            den = fmaf(exp2f(ml.x - Ms), ml.y, den);
        }
        const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll 1
        for (int c = c0; c < c0 + nc; c++) {
            if (c * 32 >= D) break;                             // warp-uniform
            uint32_t v[32];
            tmem_ld32(to + c * 32, v);
            tmem_ld_wait();
            if (!valid || !ok) continue;
            float acc[32];
#pragma unroll
            for (int k = 0; k < 32; k++) acc[k] = __uint_as_float(v[k]) * w0;
            for (int q = 0; q < pieces; q++) {
                if (q == piece) continue;
                const size_t prow = (slot0 + q) * 256 + rr;
                const float w = exp2f(__ldcg(&p.part_ml[prow]).x - Ms);
                const float4 *src = reinterpret_cast<const float4 *>(p.part_o + prow * D + c * 32);
                float4 x[8];
#pragma unroll
                for (int k = 0; k < 8; k++)
                    if (c * 32 + k * 4 < D) x[k] = __ldcg(src + k);
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    if (c * 32 + k * 4 >= D) break;
                    acc[4 * k] = fmaf(w, x[k].x, acc[4 * k]);
                    acc[4 * k + 1] = fmaf(w, x[k].y, acc[4 * k + 1]);
                    acc[4 * k + 2] = fmaf(w, x[k].z, acc[4 * k + 2]);
                    acc[4 * k + 3] = fmaf(w, x[k].w, acc[4 * k + 3]);
                }
            }
            uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow * D + c * 32);
#pragma unroll
            for (int k = 0; k < 4; k++) {
                if (c * 32 + k * 8 >= D) break;
                dst[k] = make_uint4(pack_bf16x2(acc[8 * k] * inv, acc[8 * k + 1] * inv),
                                    pack_bf16x2(acc[8 * k + 2] * inv, acc[8 * k + 3] * inv),
                                    pack_bf16x2(acc[8 * k + 4] * inv, acc[8 * k + 5] * inv),
                                    pack_bf16x2(acc[8 * k + 6] * inv, acc[8 * k + 7] * inv));
            }
        }
    }
    named_bar_sync(7, 256);
    if (threadIdx.x == 128) {                                   // ready for the next call
        atomicExch(cnt, 0u);
        atomicExch(cnt + 1, 0u);
    }
}

// A decode CTA of a mixed launch: each of its 12 warps runs decode items of
// list dl (parameters pd) over its own ring, items dealt round-robin over
// all warps of all decode CTAs (cta: this CTA's index among them).  The
// warps are independent: nothing is shared but the CTA's shared memory,
// split into one ring per warp; a warp leaves once its items are done, with
// no copy in flight.  FP8: the pool holds E4M3 codes and scales.
template <int DP, int D, bool FP8>
__device__ __forceinline__ void tc_decode_cta(const AttnParams &pd, const WorkList &dl, int cta, int ctas,
                                              const DecodeMaps &maps)
{
    using C = TcCfg<DP>;
    constexpr int NS = FP8 ? C::kDecStagesF8 : C::kDecStages;
    constexpr int kRing = FP8 ? C::kDecRingF8 : C::kDecRing;
    constexpr int kBarOff = FP8 ? C::kDecBarOffF8 : C::kDecBarOff;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t *sp = smem_raw + (sb - raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kWarps = kTcThreads / 32;
    WarpPipe wp;
    wp.ring = sb + warp * kRing;
    wp.bars = sb + kBarOff + warp * NS * 8;
    wp.stage_ptr = sp + warp * kRing;
    wp.scales = 0u;
    wp.scale_f = nullptr;
    if constexpr (FP8) {
        constexpr int kScales = NS * WarpRingF8::kScaleStage;
        wp.scales = sb + C::kDecScaleOffF8 + warp * kScales;
        wp.scale_f = reinterpret_cast<const float *>(sp + C::kDecScaleOffF8 + warp * kScales);
    }
    wp.seq = 0;
    if (lane == 0) {
        prefetch_tmap(&maps.k);
        prefetch_tmap(&maps.v);
        for (int s = 0; s < NS; s++) mbar_init(wp.bars + 8u * s, 1);
        fence_mbar_init();
    }
    __syncwarp();
    pdl_wait();                                                    // the step's earlier kernels are done
    const int items = dl.item_off[dl.n];
    for (int it = cta * kWarps + warp; it < items; it += ctas * kWarps) {
        warp_decode_item<DP, D, NS, FP8>(pd, dl, it, wp, maps);
        __syncwarp();
        // the epilogue's reads of the ring precede the next item's copies into it
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
}

// DP: head dim padded to the 64-column sub-tile; D: head dim of q and out;
// WIN: a sliding window is set (p.window > 0).  MIX: a mixed batch (0:
// none, kMixBf16 or kMixFp8: decodes over a bf16 or a quantized pool): the
// first mix->dec_rows grid rows are decode CTAs (list dl, parameters pd,
// the pool's maps dm), the tcgen05 prefill CTAs follow.
constexpr int kMixBf16 = 1, kMixFp8 = 2;
// Warps 3 .. 11 write a single-CTA request's new rows (combined call).
constexpr uint32_t kOwnRowWarps = 9;

// The new rows of request r (t tokens at positions L - t .. L - 1, token
// rows b ..) of KV head kh into the pools at fw_slots[row], as
// fused_kv_write does (a negative slot: the scratch slot; one outside the
// pool: skipped, bit 1; one other than the block table's: kDevErrMeta), by
// threads tid of nthreads.  A thread loads its rows' K and V before their
// slot, so its loads overlap; it fences its stores against the async proxy.
template <int D>
__device__ __forceinline__ void tc_own_rows(const AttnParams &p, int r, int b, int t, int L, int kh, int tid,
                                            int nthreads)
{
    constexpr int kVec = D * 2 / 16;                      // 16-byte vectors of one row and head
    const int64_t num_slots = (int64_t)p.nb_total * p.block_size;
    const int32_t *bt = p.block_table + (size_t)r * p.bt_stride;
    for (int idx = tid; idx < t * kVec; idx += nthreads) {
        const int i = idx / kVec, c = idx - i * kVec;
        const int row = b + i, pos = L - t + i;
        const size_t src = ((size_t)row * p.hkv + kh) * kVec + c;
        const uint4 kx = p.fw_k[src], vx = p.fw_v[src];
        int64_t slot = __ldg(p.fw_slots + row);
        if (c == 0 && slot >= 0) {
            const int64_t want = (int64_t)__ldg(bt + (pos >> 4)) * 16 + (pos & 15);
            if (slot != want) atomicOr(p.err, kDevErrMeta);
        }
        if (slot < 0) slot = num_slots - 1;               // padding row -> scratch slot
        if (slot >= num_slots) {
            if (c == 0) atomicOr(p.err, 1u);
            continue;
        }
        const size_t dst = ((size_t)slot * p.hkv + kh) * kVec + c;
        p.fw_kc[dst] = kx;
        p.fw_vc[dst] = vx;
    }
    fence_proxy_async_global();
}

template <int DP, int D, bool WIN, int MIX, bool OWN>
__device__ __forceinline__ void attn_tc_body(const AttnParams &p, const WorkList &wl, const CUtensorMap &qmap,
                                             const CUtensorMap &kmap, const CUtensorMap &vmap, int64_t num_slots,
                                             const AttnParams *pd, const WorkList *dl, const MixAssign *mix,
                                             const DecodeMaps *dm)
{
    if constexpr (MIX != 0) {
        if ((int)blockIdx.y < mix->dec_rows) {
            tc_decode_cta<DP, D, MIX == kMixFp8>(*pd, *dl, blockIdx.y * gridDim.x + blockIdx.x,
                                                 mix->dec_rows * gridDim.x, *dm);
            return;
        }
    }
    const int row = MIX != 0 ? (int)blockIdx.y - mix->dec_rows : (int)blockIdx.y;   // this CTA's prefill row
    using C = TcCfg<DP>;
    constexpr int kTile = C::kTile, kQOff = C::kQOff, kKOff = C::kKOff, kVOff = C::kVOff, kBarOff = C::kBarOff;
    constexpr int kHalves = C::kHalves;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t *sp = smem_raw + (sb - raw);
    auto bar = [&](int i) { return sb + kBarOff + 8u * i; };
    constexpr int kBars = OWN ? kNumTcBars + 1 : kNumTcBars;      // kBarW after the others
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sp + kBarOff + 8 * kBars);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kh = blockIdx.x;                                     // all KV heads of an item are adjacent
    const int li = find_listed(wl, row);
    const int r = wl.req[li];
    const int b = wl.qb[li], t = wl.qt[li], L = wl.len[li];
    const int g = p.group;
    const int tt = wl.tile_tokens;                                 // tokens per tile: 128 / g
    const int npairs = (t + 2 * tt - 1) / (2 * tt);
    // longest pairs first: `whole` pairs as one CTA, then `pieces` CTAs per pair
    const int local = row - wl.item_off[li];
    const int whole = tc_split_whole(wl.tc_split[li]), small = tc_split_small(wl.tc_split[li]);
    int pair = npairs - 1 - local, piece = 0, pieces = 1;
    if (local >= whole) {                                          // piece-major over the split pairs
        pieces = tc_split_pieces(wl.tc_split[li]);
        pair = npairs - 1 - whole - (local - whole) % (npairs - whole);
        piece = (local - whole) / (npairs - whole);
    }
    const int i0 = pair * 2 * tt;                                  // first token of tile a
    const int ntok_a = min(tt, t - i0);
    const int ntok_b = max(0, min(tt, t - i0 - tt));
    const bool has_b = ntok_b > 0;
    const int k_end = L - t + i0 + ntok_a + ntok_b;                // one past the last position
    // the pair's key tiles start at the one holding the window start of its
    // first row; this CTA takes key tiles jt0 .. jt0 + nkt - 1 of them
    const int jt_first = window_lo(L - t + i0, p.window) / kTcKeys;
    const int nkt_pair = (k_end + kTcKeys - 1) / kTcKeys - jt_first;
    const int jt0 = jt_first + tc_piece_begin(nkt_pair, piece, pieces, small);
    const int nkt = jt_first + tc_piece_begin(nkt_pair, piece + 1, pieces, small) - jt0;
    const int nblk = min((k_end + 15) >> 4, (jt0 + nkt) * 8) - jt0 * 8;   // blocks of those key tiles
    // split pieces: the pair's partial slots (one per piece) and counter
    const int split_idx = npairs - 1 - whole - pair;
    const size_t slot0 =
        pieces > 1 ? (size_t)wl.part_off[li] + ((size_t)split_idx * p.hkv + kh) * pieces : 0;
    uint32_t *const piece_cnt =
        pieces > 1 ? p.counters + (size_t)(wl.cnt_off[li] + split_idx * p.hkv + kh) * kCounterStride : nullptr;
    uint32_t *const s_piece = tmem_slot + 1;                       // two flag words after the TMEM address
    const int wspan = win_span(p.window);                          // keys <= position - wspan are outside
    // Combined call (p.fw_k set): a request whose rows of this KV head are
    // all one CTA's (a single pair, uncut) has its new rows written by that
    // CTA's warps 3 .. 11, not by a scatter ahead of the launch; the
    // producers wait for them before the first key tile that holds one.
    const bool self_write = OWN && p.fw_k != nullptr && npairs == 1 && pieces == 1;
    [[maybe_unused]] const int first_new_tile = (L - t) / kTcKeys; // key tile of position L - t

    if (threadIdx.x == 0) {
        // P of tile a comes from 8 warps when a single tile splits its rows;
        // that tile then alternates P(j) between kBarPA (even j) and kBarPB
        // (odd j): a warp may start tile j+1 (its S is double-buffered)
        // before every warp has arrived for tile j
        for (int i = 0; i < kNumTcBars; i++)
            mbar_init(bar(i), (i == kBarPA || i == kBarPB) ? (has_b ? 4u : 8u) : 1u);
        if constexpr (OWN) mbar_init(bar(kBarW), kOwnRowWarps);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if constexpr (OWN) {
        if (self_write && warp >= 3) {
            // -------------------------------------------------------- own rows (combined call)
            // warp 3 and the softmax warps, which have nothing to do before
            // the first S: the request's new rows of this KV head into the pool
            pdl_wait();                                            // k, v and slot_mapping come from before
            tc_own_rows<D>(p, r, b, t, L, kh, threadIdx.x - 96, kOwnRowWarps * 32);
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarW));
        }
    }

    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ TMA producers
        // warp 0 loads Q and the K tiles, warp 2 the V tiles.  A tile's
        // 8 x kHalves boxes (8 blocks x its 64-column halves) are issued by
        // as many lanes at once.
        const bool is_k = warp == 0;
        if (lane == 0) {
            if (is_k) {
                prefetch_tmap(&qmap);
                prefetch_tmap(&kmap);
                mbar_arrive_expect_tx(bar(kBarQ), has_b ? 2 * kTile : kTile);
#pragma unroll
                for (int hf = 0; hf < kHalves; hf++) {
                    tma_load_3d(sb + kQOff + hf * kSub, &qmap, bar(kBarQ), hf * 64, kh * g, b + i0);
                    if (has_b) tma_load_3d(sb + kQOff + kTile + hf * kSub, &qmap, bar(kBarQ), hf * 64, kh * g, b + i0 + tt);
                }
            } else {
                prefetch_tmap(&vmap);
            }
        }
        const CUtensorMap *map = is_k ? &kmap : &vmap;
        const uint32_t ring = sb + (is_k ? kKOff : kVOff);
        const int full0 = is_k ? kBarK0 : kBarV0;
        // A K stage is free once the last S MMA that reads it is done, a V
        // stage once the last PV MMA is: wait on those MMAs' own completion
        // barriers (their next completion needs a tile not loaded yet).
        const int done_bar = is_k ? (has_b ? kBarSB : kBarSA) : (has_b ? kBarOB : kBarOA);
        const int32_t *bt = p.block_table + (size_t)r * p.bt_stride + jt0 * 8;
        // this lane's box (lanes 0 .. 8 * kHalves - 1): block bi, column half
        const int bi = kHalves == 2 ? (lane >> 1) & 7 : lane & 7, half = kHalves == 2 ? lane & 1 : 0;
        // the block table is not written by the step's K/V scatter: the first
        // 32 block ids are read while that kernel may still be running
        int ids = lane < nblk ? __ldg(bt + lane) : INT_MIN, issued = 0;
        pdl_wait();                                                // the step's K/V rows are in the pool
        [[maybe_unused]] bool rows_in = !self_write;
        for (int j = 0; j < nkt; j++) {
            const int st = j & 1;
            if ((j & 3) == 0 && j > 0) {                           // 32 block ids = 4 key tiles
                const int jb = j * 8 + lane;
                ids = jb < nblk ? __ldg(bt + jb) : INT_MIN;
            }
            // slot row of this lane's block (beyond the range: past the pool, TMA fills zeros)
            const int blk = __shfl_sync(0xffffffffu, ids, ((j & 3) << 3) + bi);
            int row = (int)num_slots;
            if (blk != INT_MIN) {
                if (blk < 0 || blk >= p.nb_total) {
                    if (is_k && lane < 8 * kHalves && half == 0) atomicOr(p.err, 2u);
                } else {
                    row = blk * 16;
                }
            }
            bool ok = true;
            // a single tile alternates S(j) between two TMEM buffers, each
            // with its own barrier (kBarSA for even j, kBarSB for odd j)
            if (j >= 2)
                ok = (is_k && !has_b) ? mbar_wait(bar(kBarSA + (j & 1)), ((j - 2) >> 1) & 1, p.err)
                                      : mbar_wait(bar(done_bar), (j - 2) & 1, p.err);
            if constexpr (OWN) {
                if (!rows_in && jt0 + j >= first_new_tile) {       // this tile holds new rows: wait for them
                    ok = mbar_wait(bar(kBarW), 0, p.err) && ok;
                    fence_proxy_async_global();
                    rows_in = true;
                }
            }
            if (!__all_sync(0xffffffffu, ok)) break;
            issued = j + 1;
            if (lane == 0) mbar_arrive_expect_tx(bar(full0 + st), kTile);
            __syncwarp();
            if (lane < 8 * kHalves)
                tma_load_3d(ring + st * kTile + half * kSub + bi * 2048, map, bar(full0 + st), half * 64, kh, row);
            __syncwarp();
        }
        if (issued < nkt && lane == 0) {                           // a wait gave up: drain own copies
            if (is_k) mbar_wait(bar(kBarQ), 0, p.err);
            for (int j = issued > 2 ? issued - 2 : 0; j < issued; j++)
                mbar_wait(bar(full0 + (j & 1)), (j >> 1) & 1, p.err);
        }
        if (!is_k && lane == 0 && kh == 0 && row == wl.item_off[li]) check_meta(p, wl, li);
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16(kTcRows, kTcKeys, false);
            constexpr uint32_t idO = idesc_bf16(kTcRows, DP, true);
            const int ntile = has_b ? 2 : 1;
            auto issue_s = [&](int x, int j) {                     // S_x(j) = Q_x K_j^T
                const uint32_t kbase = sb + kKOff + (j & 1) * kTile;
                const uint32_t qbase = sb + kQOff + x * kTile;
#pragma unroll
                for (int kk = 0; kk < DP / 16; kk++) {
                    const uint64_t ad = sdesc_sw128(qbase + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(kbase + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024);
                    tc_mma(tmem + x * 128, ad, bd, idS, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(kBarSA + x));
            };
            auto issue_pv = [&](int x, int i) -> bool {            // O_x += P_x(i) V_i
                if (!mbar_wait(bar(kBarPA + x), i & 1, p.err)) return false;
                if (x == 0 && !mbar_wait(bar(kBarV0 + (i & 1)), (i >> 1) & 1, p.err)) return false;
                tc_fence_after();
                const uint32_t vbase = sb + kVOff + (i & 1) * kTile;
#pragma unroll
                for (int kk = 0; kk < 8; kk++) {
                    const uint64_t bd = sdesc_sw128(vbase + kk * 2048, kSub, 1024);
                    tc_mma_ts(tmem + 256 + x * 128, tmem + x * 128 + kk * 8, bd, idO, (i > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar(kBarOA + x));
                return true;
            };
            auto issue_s1 = [&](int j) {                          // single tile: S(j) into buffer j & 1
                const uint32_t kbase = sb + kKOff + (j & 1) * kTile;
#pragma unroll
                for (int kk = 0; kk < DP / 16; kk++) {
                    const uint64_t ad = sdesc_sw128(sb + kQOff + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(kbase + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024);
                    tc_mma(tmem + (j & 1) * 128, ad, bd, idS, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(kBarSA + (j & 1)));
            };
            auto issue_pv1 = [&](int j) -> bool {                  // single tile: O += P(j) V_j
                if (!mbar_wait(bar(kBarPA + (j & 1)), (j >> 1) & 1, p.err)) return false;
                if (!mbar_wait(bar(kBarV0 + (j & 1)), (j >> 1) & 1, p.err)) return false;
                tc_fence_after();
                const uint32_t vbase = sb + kVOff + (j & 1) * kTile;
#pragma unroll
                for (int kk = 0; kk < 8; kk++) {
                    const uint64_t bd = sdesc_sw128(vbase + kk * 2048, kSub, 1024);
                    // P of keys 0..63 at columns [0,32), of keys 64..127 at [64,96)
                    const uint32_t pcol = (j & 1) * 128 + kk * 8 + (kk >= 4 ? 32 : 0);
                    tc_mma_ts(tmem + 256, tmem + pcol, bd, idO, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar(kBarOA));
                return true;
            };
            bool ok = mbar_wait(bar(kBarQ), 0, p.err);
            if (has_b) {
                for (int j = 0; j < nkt && ok; j++) {
                    for (int x = 0; x < ntile && ok; x++) {
                        if (j >= 1) ok = issue_pv(x, j - 1);     // reads P_x(j-1) before S_x(j) overwrites it
                        if (ok && x == 0) {
                            ok = mbar_wait(bar(kBarK0 + (j & 1)), (j >> 1) & 1, p.err);
                            tc_fence_after();
                        }
                        if (ok) issue_s(x, j);
                    }
                }
                for (int x = 0; x < ntile && ok; x++) ok = issue_pv(x, nkt - 1);
            } else {
                // single tile: S(j) goes to TMEM columns [128 (j & 1), +128)
                // and completes on barrier kBarSA + (j & 1), so S(j+1) runs
                // while the softmax of tile j does; PV(j) reads P(j) there
                // before S(j+2) overwrites it (MMAs complete in issue order)
                for (int j = 0; j < nkt && ok; j++) {
                    if (j == 0) {
                        ok = mbar_wait(bar(kBarK0), 0, p.err);
                        tc_fence_after();
                        if (ok) issue_s1(0);
                    }
                    if (ok && j + 1 < nkt) {
                        ok = mbar_wait(bar(kBarK0 + ((j + 1) & 1)), ((j + 1) >> 1) & 1, p.err);
                        tc_fence_after();
                        if (ok) issue_s1(j + 1);
                    }
                    if (ok) ok = issue_pv1(j);
                }
                // With S double-buffered, S(j) does not imply PV(j-1) done,
                // so kBarOA may lag its waiters by two phases at the end: the
                // final O gets its own single-phase barrier.
                tc_commit(bar(kBarOFin));
            }
            // every MMA this thread issued has finished before TMEM is released
            tc_commit(bar(kBarMmaDone));
            mbar_wait(bar(kBarMmaDone), 0, p.err);
        }
        __syncwarp();
    } else if (warp >= 4 && has_b) {
        // ------------------------------------------------------------ softmax, one row per thread
        const int x = warp >= 8 ? 1 : 0;                           // tile a or b
        const int row = threadIdx.x - (x ? 256 : 128);
        const int ntok_x = x ? ntok_b : ntok_a;
        const int nr = ntok_x * g;
        const int tok0 = i0 + x * tt;                              // first token of this tile
        const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t ts = tl + x * 128;                          // S_x (and P_x) columns
        const uint32_t to = tl + 256 + x * 128;                    // O_x columns
        const int qpos = row < nr ? L - t + tok0 + row / g : -1;
        const int qlo = qpos - wspan;                              // keys at or below are outside the window
        const float sl2 = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkt; j++) {
            ok = mbar_wait(bar(kBarSA + x), j & 1, p.err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            const int key0 = (jt0 + j) * kTcKeys;
            // warp-uniform: does any row of this warp see masked keys in this tile?
            const bool diag = __any_sync(0xffffffffu, key0 + kTcKeys - 1 > qpos || (WIN && key0 <= qlo));
            const float mraw = diag ? tc_row_max<true, 128, WIN>(ts, key0, qpos, qlo) : tc_row_max<false, 128, WIN>(ts, key0, qpos, qlo);
            const float mt = mraw * sl2;                            // in the exp2 domain (scale > 0)
            if (j == 0) {
                m_used = mt;
            } else {
                const bool need = mt > m_used + kRescaleLog2;
                if (__any_sync(0xffffffffu, need)) {
                    // move the running max: O_x must be stable, so wait for PV_x(j-1)
                    ok = mbar_wait(bar(kBarOA + x), (j - 1) & 1, p.err);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    tc_fence_after();
                    const float alpha = need ? exp2f(m_used - mt) : 1.f;
                    if (need) {
                        l *= alpha;
                        m_used = mt;
                    }
                    tc_rescale_cols(to, 0, DP / 32, alpha);
                }
            }
            // pass 2: P = 2^(s * scale * log2e - m) over the first 64 S columns
            const float ms = m_used == -INFINITY ? 0.f : m_used;
            l += diag ? tc_row_exp<true, 128, WIN>(ts, key0, qpos, qlo, sl2, ms) : tc_row_exp<false, 128, WIN>(ts, key0, qpos, qlo, sl2, ms);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarPA + x));
        }
        pdl_launch_dependents();
        if (ok) ok = mbar_wait(bar(kBarOA + x), (nkt - 1) & 1, p.err);
        ok = __all_sync(0xffffffffu, ok);
        if (ok) tc_fence_after();
        if (pieces > 1) {
            const size_t orow = row < nr ? (size_t)(b + tok0 + row / g) * p.hq + kh * g + row % g : 0;
            tc_piece_epilogue<D>(p, piece_cnt, slot0, piece, pieces, to, x * 128 + row, row < nr, m_used, l, 0,
                                 DP / 32, true, ok, orow, s_piece);
        } else if (ok) {
            tc_store_rows<D>(p, to, row, nr, b + tok0, kh, g, l > 0.f ? 1.f / l : 0.f, 0, DP / 32);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ single tile: two warps per row
        // Warps w and w + 4 share TMEM lanes 32 (w % 4) ..: warp hc = 0 takes
        // S columns [0,64) and O columns [0,DP/2), hc = 1 the other halves.
        // Each pair meets at a named barrier per key tile (ids 2..5) to swap
        // half-row maxima; it ANDs the pair's progress so both leave together.
        const int hc = warp >= 8 ? 1 : 0;
        const int rg = warp & 3;
        const int row = threadIdx.x - (hc ? 256 : 128);
        const int nr = ntok_a * g;
        const uint32_t tl = tmem + ((uint32_t)(rg * 32) << 16);
        const uint32_t to = tl + 256;                              // O_a
        const int qpos = row < nr ? L - t + i0 + row / g : -1;
        const int qlo = qpos - wspan;                              // keys at or below are outside the window
        const float sl2 = p.scale_log2;
        float *xm = reinterpret_cast<float *>(sp + C::kXOff);      // [parity][half][128]
        float *xl = xm + 512;                                      // [half][128]
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkt; j++) {
            const uint32_t ts = tl + (j & 1) * 128 + hc * 64;     // this half of S(j); P at its first 32 columns
            ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarSA + (j & 1)), (j >> 1) & 1, p.err));
            const int key0 = (jt0 + j) * kTcKeys + hc * 64;
            const bool diag = __any_sync(0xffffffffu, key0 + 63 > qpos || (WIN && key0 <= qlo));
            float mh = -INFINITY;
            if (ok) {
                tc_fence_after();
                mh = diag ? tc_row_max<true, 64, WIN>(ts, key0, qpos, qlo) : tc_row_max<false, 64, WIN>(ts, key0, qpos, qlo);
                xm[((j & 1) * 2 + hc) * 128 + row] = mh;
            }
            if (!named_bar_and(2 + rg, 64, ok)) { ok = false; break; }
            const float mt = fmaxf(mh, xm[((j & 1) * 2 + (hc ^ 1)) * 128 + row]) * sl2;
            if (j == 0) {
                m_used = mt;
            } else {
                const bool need = mt > m_used + kRescaleLog2;       // the same in both halves
                if (__any_sync(0xffffffffu, need)) {
                    // move the running max: O must be stable, so wait for PV(j-1);
                    // both warps of the pair take this branch and agree on the outcome
                    ok = mbar_wait(bar(kBarOA), (j - 1) & 1, p.err);
                    if (!named_bar_and(2 + rg, 64, __all_sync(0xffffffffu, ok))) { ok = false; break; }
                    tc_fence_after();
                    const float alpha = need ? exp2f(m_used - mt) : 1.f;
                    if (need) {
                        l *= alpha;
                        m_used = mt;
                    }
                    tc_rescale_cols(to, hc * (DP / 64), DP / 64, alpha);
                }
            }
            const float ms = m_used == -INFINITY ? 0.f : m_used;
            l += diag ? tc_row_exp<true, 64, WIN>(ts, key0, qpos, qlo, sl2, ms) : tc_row_exp<false, 64, WIN>(ts, key0, qpos, qlo, sl2, ms);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarPA + (j & 1)));
        }
        pdl_launch_dependents();
        if (ok) ok = mbar_wait(bar(kBarOFin), 0, p.err);
        xl[hc * 128 + row] = l;
        ok = named_bar_and(2 + rg, 64, __all_sync(0xffffffffu, ok));
        if (ok) tc_fence_after();
        const float lt = l + xl[(hc ^ 1) * 128 + row];
        if (pieces > 1) {
            const size_t orow = row < nr ? (size_t)(b + i0 + row / g) * p.hq + kh * g + row % g : 0;
            tc_piece_epilogue<D>(p, piece_cnt, slot0, piece, pieces, to, row, row < nr, m_used, lt,
                                 hc * (DP / 64), DP / 64, hc == 0, ok, orow, s_piece);
        } else if (ok) {
            tc_store_rows<D>(p, to, row, nr, b + i0, kh, g, lt > 0.f ? 1.f / lt : 0.f, hc * (DP / 64), DP / 64);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// OWN: combined calls whose single-CTA requests write their own rows (a
// separate instantiation, so that the other launches' code is not touched
// by the writers' prologue).
template <int DP, int D, bool WIN, bool OWN>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(AttnParams p, const __grid_constant__ WorkList wl,
                                                                const __grid_constant__ CUtensorMap qmap,
                                                                const __grid_constant__ CUtensorMap kmap,
                                                                const __grid_constant__ CUtensorMap vmap,
                                                                int64_t num_slots)
{
    attn_tc_body<DP, D, WIN, 0, OWN>(p, wl, qmap, kmap, vmap, num_slots, nullptr, nullptr, nullptr, nullptr);
}

template <int DP, int D, bool WIN, int MIX>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_mix_kernel(AttnParams p, const __grid_constant__ WorkList wl, const __grid_constant__ CUtensorMap qmap,
                       const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                       int64_t num_slots, AttnParams pd, const __grid_constant__ WorkList dl,
                       const __grid_constant__ MixAssign mix, const __grid_constant__ DecodeMaps dm)
{
    attn_tc_body<DP, D, WIN, MIX, false>(p, wl, qmap, kmap, vmap, num_slots, &pd, &dl, &mix, &dm);
}

// ---------------------------------------------------------------- host side

cudaError_t make_pool_tmap(CUtensorMap *map, const void *pool, int64_t num_slots, int hkv, int d, int box_cols,
                           bool swizzle128);
cudaError_t make_q_tmap(CUtensorMap *map, const void *q, int num_tokens, int hq, int d, int g);
cudaError_t make_code_tmap(CUtensorMap *map, const void *pool, int64_t num_slots, int hkv);

bool tc_prefill_supported(int head_dim, int group)
{
    return (head_dim == 48 || head_dim == 64 || head_dim == 128) && group >= 1 && kTcRows % group == 0;
}
int tc_prefill_rows() { return kTcRows; }

template <int DP, int D, bool WIN>
static cudaError_t launch_tc_d(const AttnParams &p, const WorkList &wl, int num_items, const void *q, int num_tokens,
                               const void *k_cache, const void *v_cache, int64_t num_slots, cudaStream_t stream,
                               const AttnParams *pd, const WorkList *dl, const MixAssign *mix)
{
    constexpr int smem = TcCfg<DP>::kSmem, smem_mix = TcCfg<DP>::kSmemMix, smem_f8 = TcCfg<DP>::kSmemMixF8;
    constexpr bool kHasF8 = DP == 128 && D == 128;                 // quantized pools: head dim 128
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(attn_tc_kernel<DP, D, WIN, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        smem);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(attn_tc_kernel<DP, D, WIN, true>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (attr_err == cudaSuccess)
            attr_err = cudaFuncSetAttribute(attn_tc_mix_kernel<DP, D, WIN, kMixBf16>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, smem_mix);
        if (attr_err == cudaSuccess && kHasF8)
            attr_err = cudaFuncSetAttribute(attn_tc_mix_kernel<DP, D, WIN, kHasF8 ? kMixFp8 : kMixBf16>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, smem_f8);
    });
    if (attr_err != cudaSuccess) return attr_err;
    const bool fp8_dec = mix && pd->k_scale != nullptr;
    if (fp8_dec && !kHasF8) return cudaErrorInvalidValue;
    if (mix && p.fw_k) return cudaErrorInvalidValue;                // a mixed launch's chunks come from the scatter
    CUtensorMap qm, km, vm;
    // 64-column boxes; for D < 64 they reach past the row and TMA fills zeros
    cudaError_t e = make_q_tmap(&qm, q, num_tokens, p.hq, D, p.group);
    if (e == cudaSuccess) e = make_pool_tmap(&km, k_cache, num_slots, p.hkv, D, 64, true);
    if (e == cudaSuccess) e = make_pool_tmap(&vm, v_cache, num_slots, p.hkv, D, 64, true);
    if (e != cudaSuccess) return e;
    // the decode items' pool: the prefill's own (bf16), or the quantized
    // pool whose bf16 copies the prefill reads
    DecodeMaps dm;
    if (mix) {
        if (fp8_dec) {
            const int64_t dslots = (int64_t)pd->nb_total * 16;
            e = make_code_tmap(&dm.k, pd->k_cache, dslots, pd->hkv);
            if (e == cudaSuccess) e = make_code_tmap(&dm.v, pd->v_cache, dslots, pd->hkv);
            if (e != cudaSuccess) return e;
        } else {
            dm.k = km;
            dm.v = vm;
        }
    }
    const int rows = num_items + (mix ? mix->dec_rows : 0);
    if (rows > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid(p.hkv, rows);                        // items in launch order: the planner puts the longest first
    launch_begin(stream, mix ? kAttnTcMixed : kAttnTcPrefill);
    if (fp8_dec)
        e = launch_maybe_pdl(attn_tc_mix_kernel<DP, D, WIN, kHasF8 ? kMixFp8 : kMixBf16>, grid, dim3(kTcThreads),
                             smem_f8, stream, p, wl, qm, km, vm, num_slots, *pd, *dl, *mix, dm);
    else if (mix)
        e = launch_maybe_pdl(attn_tc_mix_kernel<DP, D, WIN, kMixBf16>, grid, dim3(kTcThreads), smem_mix, stream, p,
                             wl, qm, km, vm, num_slots, *pd, *dl, *mix, dm);
    else if (p.fw_k)
        e = launch_maybe_pdl(attn_tc_kernel<DP, D, WIN, true>, grid, dim3(kTcThreads), smem, stream, p, wl, qm, km,
                             vm, num_slots);
    else
        e = launch_maybe_pdl(attn_tc_kernel<DP, D, WIN, false>, grid, dim3(kTcThreads), smem, stream, p, wl, qm, km,
                             vm, num_slots);
    launch_end(stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_attn_tc(const AttnParams &p, const WorkList &wl, int num_items, const void *q, int num_tokens,
                           const void *k_cache, const void *v_cache, int64_t num_slots, int head_dim,
                           cudaStream_t stream, const AttnParams *pd, const WorkList *dl, const MixAssign *mix)
{
    if (num_items <= 0) return cudaSuccess;
    if (mix && (!pd || !dl || mix->dec_rows <= 0)) return cudaErrorInvalidValue;
    const bool win = p.window > 0;
#define PKV_TC_ARGS p, wl, num_items, q, num_tokens, k_cache, v_cache, num_slots, stream, pd, dl, mix
    switch (head_dim) {
    case 48: return win ? launch_tc_d<64, 48, true>(PKV_TC_ARGS) : launch_tc_d<64, 48, false>(PKV_TC_ARGS);
    case 64: return win ? launch_tc_d<64, 64, true>(PKV_TC_ARGS) : launch_tc_d<64, 64, false>(PKV_TC_ARGS);
    case 128: return win ? launch_tc_d<128, 128, true>(PKV_TC_ARGS) : launch_tc_d<128, 128, false>(PKV_TC_ARGS);
    default: return cudaErrorInvalidValue;
    }
#undef PKV_TC_ARGS
}

}  // namespace pkv

// Warp-level MMA tiles over staged KV block slices, shared by the decode
// kernels and the tcgen05 prefill kernel's decode warps.
//
// A K or V slice is the 16 rows of one paged block for one KV head ("31.
// Engine v2", "Attention over the pool": key j lives in block table[j / 16],
// row j % 16), copied by TMA into shared memory: for head_dim 64/128 (bf16)
// as boxes of 16 rows x 64 columns (128 bytes) with the 128-byte swizzle, so
// that ldmatrix reads eight rows without bank conflicts; for head_dim 48 as
// unswizzled 96-byte rows.
#pragma once

#include "common.cuh"
#include "sm100.cuh"

namespace pkv {

// Quantized pools: FP8 E4M3 K/V (one byte per element) with an fp32 scale
// per (slot, KV head).  A block's scales are staged with it as one 2-D TMA
// box of 16 slots x the 4 KV heads of the CTA's group of four (256 bytes).
constexpr int kScaleHeads = 4;

template <int D, bool FP8 = false>
struct MmaTile {
    static constexpr int kElem = FP8 ? 1 : 2;
    static constexpr int kRowBytes = D * kElem;
    static constexpr bool kSwizzle = kRowBytes % 128 == 0;   // rows of 128-byte boxes, 128-byte swizzle
    static constexpr int kBoxCols = kSwizzle ? 128 / kElem : D;   // columns per TMA box
    static constexpr int kBoxes = D / kBoxCols;              // boxes per 16-row slice
    static constexpr int kBoxBytes = 16 * kBoxCols * kElem;
    static constexpr int kTile = 16 * kRowBytes;             // one K (or V) slice
    static constexpr int kScaleTile = FP8 ? 16 * kScaleHeads * 4 : 0;  // [16 slots][4 heads] fp32
    static constexpr int kData = 2 * kTile + 2 * kScaleTile; // K, V, K scales, V scales
    // one-block ring slots keep swizzled tiles on 1024-byte boundaries
    static constexpr int kSlot = kSwizzle ? (kData + 1023) / 1024 * 1024 : kData;
};

// Byte offset of 16-byte chunk `chunk` of row `row` inside a K or V slice.
template <int D, bool FP8 = false>
__device__ __forceinline__ uint32_t tile_off(int row, int chunk)
{
    if constexpr (!MmaTile<D, FP8>::kSwizzle) {
        return row * MmaTile<D, FP8>::kRowBytes + chunk * 16;
    } else {
        const int box = chunk >> 3, c = chunk & 7;
        return box * 2048 + row * 128 + ((c ^ (row & 7)) << 4);
    }
}

// ---------------------------------------------------------------- key-major decode tiles
//
// A decode CTA holds few rows (t * g <= 8 pairs of (token, query head) per
// KV head: 2, 4 and 8 on the decode workloads), so a 16-row MMA tile of
// query rows is mostly padding.  The transposed products put the 16 keys of
// a block (or 16 head dims) in the MMA's M dimension and up to 8 rows in N:
//   S^T  = K Q^T        m16 keys      x n8 rows x k16 head dims
//   O^T += V^T P^T      m16 head dims x n8 rows x k16 keys
// which halves the MMAs per block.  Lane 4r + c holds S^T for keys r and
// r + 8 of the block and rows 2c, 2c + 1; a movmatrix of each 8-key half of
// P^T gives the B fragments of the second product.  O^T tile mt holds, for
// rows 2c, 2c + 1, head dims ot_dim(mt, r, 0) and ot_dim(mt, r, 1).
constexpr int kKeyMajorRows = 8;

// Q^T as m16n8k16 B fragments: lane 4r + c holds row r (zero when r >= the
// CTA's rows).  bf16: dims 2c, 2c+1 and 2c+8, 2c+9 of every 16-dim chunk;
// FP8 pools: dims 4c .. 4c+3 (the order an ldmatrix of FP8 K rows gives, as
// in load_q_frags), converted to fp16.
template <int D, bool FP8>
__device__ __forceinline__ void load_qt_frags(uint32_t (&qb)[D / 16][2], const __nv_bfloat16 *q, size_t row, bool ok,
                                              int lane)
{
    const int c = lane & 3;
    if constexpr (!FP8) {
        const uint32_t *qw = reinterpret_cast<const uint32_t *>(q);
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
            qb[kk][0] = ok ? __ldg(qw + row * (D / 2) + kk * 8 + c) : 0u;
            qb[kk][1] = ok ? __ldg(qw + row * (D / 2) + kk * 8 + 4 + c) : 0u;
        }
    } else {
        const uint2 *q4 = reinterpret_cast<const uint2 *>(q);      // 4 bf16 per load
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
            const uint2 a = ok ? __ldg(q4 + row * (D / 4) + kk * 4 + c) : make_uint2(0u, 0u);
            qb[kk][0] = pack_f16x2(bf16_lo(a.x), bf16_hi(a.x));
            qb[kk][1] = pack_f16x2(bf16_lo(a.y), bf16_hi(a.y));
        }
    }
}

// S^T for one 16-key block (accumulated into s; two chains over alternate
// head-dim chunks).  FP8: K codes converted to fp16 (exact); the K scales
// are applied by the caller.
// HP > 1 (FP8 pools): the slice holds the rows of HP adjacent KV heads
// interleaved (row r of head hd at slice row r * HP + hd, as a TMA box of HP
// heads lays them out); hd selects the head.
template <int D, bool FP8, int HP = 1>
__device__ __forceinline__ void block_scores_t(float (&s)[4], const uint32_t (&qb)[D / 16][2], uint32_t kt, int mi,
                                               int mr, int hd = 0)
{
    static_assert(HP == 1 || FP8, "interleaved heads: FP8 pools only");
    float s1[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (!FP8) {
        // matrix mi: keys (mi & 1) * 8 .., dims of half mi >> 1 of the chunk
#pragma unroll
        for (int kk = 0; kk < D / 16; kk++) {
            uint32_t a[4];
            ldsm_x4(kt + tile_off<D>((mi & 1) * 8 + mr, 2 * kk + (mi >> 1)), a[0], a[1], a[2], a[3]);
            if (kk & 1) mma_16816(s1, a, qb[kk][0], qb[kk][1]);
            else mma_16816(s, a, qb[kk][0], qb[kk][1]);
        }
    } else {
        // matrix mi: keys (mi & 1) * 8 .., 16-code chunk kk + (mi >> 1); a
        // lane gets codes 4c .. 4c+3 of one key
#pragma unroll
        for (int kk = 0; kk < D / 16; kk += 2) {
            uint32_t r0, r1, r2, r3, a[4], a2[4];
            ldsm_x4(kt + tile_off<D, true>(((mi & 1) * 8 + mr) * HP + hd, kk + (mi >> 1)), r0, r1, r2, r3);
            e4m3x4_to_f16x2x2(r0, a[0], a[2]);
            e4m3x4_to_f16x2x2(r1, a[1], a[3]);
            e4m3x4_to_f16x2x2(r2, a2[0], a2[2]);
            e4m3x4_to_f16x2x2(r3, a2[1], a2[3]);
            mma_16816_f16(s, a, qb[kk][0], qb[kk][1]);
            mma_16816_f16(s1, a2, qb[kk + 1][0], qb[kk + 1][1]);
        }
    }
#pragma unroll
    for (int v = 0; v < 4; v++) s[v] += s1[v];
}

// Head dim of O^T tile mt, M-row r (hi = 0) or r + 8 (hi = 1).  FP8 pools:
// tiles 2q and 2q + 1 hold the even and the odd dims of 16-dim chunks 2q
// (rows 0-7) and 2q + 1 (rows 8-15), from the byte permute in block_pv_t.
template <bool FP8>
__device__ __forceinline__ int ot_dim(int mt, int r, int hi)
{
    return FP8 ? 16 * ((mt & ~1) + hi) + 2 * r + (mt & 1) : 16 * mt + 8 * hi + r;
}

// O^T += V^T P^T for one 16-key block; pb0 / pb1 = P^T for keys 2c, 2c+1 /
// 2c+8, 2c+9 of row r.  HP, hd: interleaved heads, as in block_scores_t.
template <int D, bool FP8, int HP = 1>
__device__ __forceinline__ void block_pv_t(float (&o)[D / 16][4], uint32_t pb0, uint32_t pb1, uint32_t vt, int mi,
                                           int mr, int hd = 0)
{
    static_assert(HP == 1 || FP8, "interleaved heads: FP8 pools only");
    if constexpr (!FP8) {
        // matrix mi: keys (mi >> 1) * 8 .., dims of half mi & 1 of tile mt;
        // transposed, a lane gets keys 2c, 2c+1 of one dim
#pragma unroll
        for (int mt = 0; mt < D / 16; mt++) {
            uint32_t a[4];
            ldsm_x4_t(vt + tile_off<D>((mi >> 1) * 8 + mr, 2 * mt + (mi & 1)), a[0], a[1], a[2], a[3]);
            mma_16816(o[mt], a, pb0, pb1);
        }
    } else {
        // matrix mi: keys (mi >> 1) * 8 .., 16-code chunk q + (mi & 1);
        // transposed, a lane gets dims 2r, 2r+1 of keys 2c, 2c+1, split by the
        // permute into the even-dim and the odd-dim fp16 pair
#pragma unroll
        for (int q = 0; q < D / 16; q += 2) {
            uint32_t r0, r1, r2, r3, ev[4], od[4];
            ldsm_x4_t(vt + tile_off<D, true>(((mi >> 1) * 8 + mr) * HP + hd, q + (mi & 1)), r0, r1, r2, r3);
            e4m3x4_to_f16x2x2(prmt(r0, 0u, 0x3120u), ev[0], od[0]);
            e4m3x4_to_f16x2x2(prmt(r1, 0u, 0x3120u), ev[1], od[1]);
            e4m3x4_to_f16x2x2(prmt(r2, 0u, 0x3120u), ev[2], od[2]);
            e4m3x4_to_f16x2x2(prmt(r3, 0u, 0x3120u), ev[3], od[3]);
            mma_16816_f16(o[q], ev, pb0, pb1);
            mma_16816_f16(o[q + 1], od, pb0, pb1);
        }
    }
}

// Scale into the exp2 domain and mask one block of S^T: s[0], s[1] are key
// `key` for rows 2c, 2c+1 (positions qp0, qp1; -1 = no row), s[2], s[3] key
// `key` + 8.  f0 / f1: the factors of the two keys.
__device__ __forceinline__ void mask_scale_t(float (&s)[4], int key, int k_end, int qp0, int qp1, int wspan, bool has,
                                             float f0, float f1)
{
#pragma unroll
    for (int v = 0; v < 4; v++) {
        const int k = key + (v >> 1) * 8;
        const int qp = (v & 1) ? qp1 : qp0;
        const bool ok = has && k < k_end && k <= qp && k > qp - wspan;
        s[v] = ok ? s[v] * ((v >> 1) ? f1 : f0) : -INFINITY;
    }
}

// Online softmax over NB blocks of masked S^T (exp2 domain), then O^T +=
// V^T P^T.  m, l: rows 2c, 2c+1 (l summed over this lane's keys only).  The
// O^T rescale is skipped when no row of the warp raised its maximum.  FP8:
// each key's V scale (vs: keys r, r+8) is folded into P, which is fp16.
template <int D, bool FP8, int NB, int HP = 1>
__device__ __forceinline__ void softmax_pv_t(float (&o)[D / 16][4], float (&m)[2], float (&l)[2], float (&s)[NB][4],
                                             const float (&vs)[NB][2], const uint32_t (&vt)[NB], const bool (&has)[NB],
                                             int mi, int mr, int hd = 0)
{
    float alpha[2];
#pragma unroll
    for (int j = 0; j < 2; j++) {
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < NB; q++) mx = max3f(mx, s[q][j], s[q][2 + j]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mnew = fmaxf(m[j], mx);
        const float ms = mnew == -INFINITY ? 0.f : mnew;
        alpha[j] = exp2f(m[j] - ms);
        m[j] = mnew;
        float sum = 0.f;
#pragma unroll
        for (int q = 0; q < NB; q++) {
            s[q][j] = exp2f(s[q][j] - ms);
            s[q][2 + j] = exp2f(s[q][2 + j] - ms);
            sum += s[q][j] + s[q][2 + j];
        }
        l[j] = l[j] * alpha[j] + sum;
    }
    if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
        for (int mt = 0; mt < D / 16; mt++) {
            o[mt][0] *= alpha[0];
            o[mt][2] *= alpha[0];
            o[mt][1] *= alpha[1];
            o[mt][3] *= alpha[1];
        }
    }
#pragma unroll
    for (int q = 0; q < NB; q++) {
        if (!has[q]) continue;
        uint32_t lo, hi;                                           // P^T [key][row] halves
        if constexpr (FP8) {
            lo = pack_f16x2(s[q][0] * vs[q][0], s[q][1] * vs[q][0]);
            hi = pack_f16x2(s[q][2] * vs[q][1], s[q][3] * vs[q][1]);
        } else {
            lo = pack_bf16x2(s[q][0], s[q][1]);
            hi = pack_bf16x2(s[q][2], s[q][3]);
        }
        block_pv_t<D, FP8, HP>(o, movmatrix_t(lo), movmatrix_t(hi), vt[q], mi, mr, hd);
    }
}

// Split-KV combine of one (request, KV head) inside the CTA that completed
// its last split.  Row (token i, head h) has S partials o_s (unnormalised),
// m_s (running max, exp2 domain) and l_s (weight sum) at rows
// base + s * t * hq + i * hq + h; the exact result is
//   o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s.
// The partials of the other splits were written by other CTAs: they are read
// through L2 (ld.global.cg), after the counter handshake's fences.
template <int D>
__device__ __forceinline__ void combine_in_cta(const AttnParams &p, size_t base, int b, int t, int kh, int g, int S,
                                               int tid, int nthreads)
{
    constexpr int kChunks = D / 8;
    const size_t rows = (size_t)t * p.hq;
    for (int idx = tid; idx < t * g * kChunks; idx += nthreads) {
        const int rr = idx / kChunks, e0 = (idx - rr * kChunks) * 8;
        const int i = rr / g, h = kh * g + (rr - (rr / g) * g);
        const size_t row = (size_t)i * p.hq + h;
        // one pass, four splits at a time: their loads go out together, then
        // each is merged into the running (M, ls, acc) with the usual rescale
        float M = -INFINITY, ls = 0.f;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int s0 = 0; s0 < S; s0 += 4) {
            float2 ml[4];
            float4 x0[4], x1[4];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                if (s0 + u < S) {
                    const size_t prow = base + (size_t)(s0 + u) * rows + row;
                    ml[u] = __ldcg(&p.part_ml[prow]);
                    const float4 *src = reinterpret_cast<const float4 *>(p.part_o + prow * D + e0);
                    x0[u] = __ldcg(src);
                    x1[u] = __ldcg(src + 1);
                } else {
                    ml[u] = make_float2(-INFINITY, 0.f);
                    x0[u] = x1[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const float Mn = fmaxf(M, ml[u].x);
                const float Ms = Mn == -INFINITY ? 0.f : Mn;
                const float a = exp2f(M - Ms), w = exp2f(ml[u].x - Ms);   // 2^-inf = 0
                ls = fmaf(ls, a, w * ml[u].y);
                acc[0] = fmaf(acc[0], a, w * x0[u].x); acc[1] = fmaf(acc[1], a, w * x0[u].y);
                acc[2] = fmaf(acc[2], a, w * x0[u].z); acc[3] = fmaf(acc[3], a, w * x0[u].w);
                acc[4] = fmaf(acc[4], a, w * x1[u].x); acc[5] = fmaf(acc[5], a, w * x1[u].y);
                acc[6] = fmaf(acc[6], a, w * x1[u].z); acc[7] = fmaf(acc[7], a, w * x1[u].w);
                M = Mn;
            }
        }
        const float inv = ls > 0.f ? 1.f / ls : 0.f;
        uint4 v;
        v.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        v.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        v.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
        v.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
        *reinterpret_cast<uint4 *>(p.out + ((size_t)(b + i) * p.hq + h) * D + e0) = v;
    }
}

}  // namespace pkv

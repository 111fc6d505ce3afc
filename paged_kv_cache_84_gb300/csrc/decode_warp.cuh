// Decode attention run by a single warp over its own ring of KV stages.
//
// The decode CTAs of a mixed tcgen05 launch run the decode-class work of
// the step: its CTAs are bound by the tensor pipe, decode attention by
// HBM, so the two share the GPU in one launch.  A decode item is one
// (request, KV head, key split) of a decode-class request (t * g <= 8 rows
// per KV head).  The warp walks the item's key blocks ("31. Engine v2",
// "Attention over the pool": key j in block table[j / 16], row j % 16),
// lane 0 issuing the TMA copies of a block's K and V slices (quantized
// pools: E4M3 codes and their per (slot, head) scales) into the next of NS
// stages, every lane computing key-major MMA tiles (S^T = K Q^T, then
// O^T += V^T P^T, online softmax in the exp2 domain: mma_tiles.cuh) as the
// stages land.  The stage count carries over from item to item (`seq`), so
// each stage's barrier keeps counting phases.
#pragma once

#include "common.cuh"
#include "mma_tiles.cuh"
#include "sm100.cuh"

namespace pkv {

// Stage layout of a warp ring for head dims padded to DP (64 or 128): the
// K slice, then the V slice, each [16][DP] bf16 as the pool's 64-column
// TMA boxes with the 128-byte swizzle lay it out.
template <int DP>
struct WarpRing {
    static constexpr int kSlice = 16 * DP * 2;
    static constexpr int kStage = 2 * kSlice;
    static constexpr int kBytes = kStage;                       // what a stage's copies deliver
};

// Stage layout of a warp ring over a quantized pool (head dim 128): the K
// codes [16][128] as one 128-byte-swizzled box, then the V codes.  The
// block's K and V scales of the item's KV head (16 fp32 each) go to a
// separate array of kScaleStage bytes per stage: the warp's lanes copy them
// with cp.async, one scale each, so that a block takes two TMA copies.
struct WarpRingF8 {
    static constexpr int kSlice = 16 * 128;
    static constexpr int kStage = 2 * kSlice;
    static constexpr int kBytes = kStage;                       // what a stage's TMA copies deliver
    static constexpr int kScaleStage = 2 * 16 * 4;
};

// Tensor maps of the pool the decode items read: K and V (boxes of 64
// bf16 columns, or 128 E4M3 codes, x 1 head x 16 slots, 128-byte swizzle).
struct DecodeMaps {
    CUtensorMap k, v;
};

// Q^T of this lane's row as B fragments for head dims padded to DP: lane
// 4r + c holds row r; dims at or past D (and rows past nr) are zero.
template <int DP, int D>
__device__ __forceinline__ void load_qt_frags_pad(uint32_t (&qb)[DP / 16][2], const __nv_bfloat16 *q, size_t row,
                                                  bool ok, int lane)
{
    const int c = lane & 3;
    const uint32_t *qw = reinterpret_cast<const uint32_t *>(q);
#pragma unroll
    for (int kk = 0; kk < DP / 16; kk++) {
        const int d0 = kk * 16 + 2 * c, d1 = d0 + 8;
        qb[kk][0] = ok && d0 < D ? __ldg(qw + row * (D / 2) + d0 / 2) : 0u;
        qb[kk][1] = ok && d1 < D ? __ldg(qw + row * (D / 2) + d1 / 2) : 0u;
    }
}

// Per-warp pipeline state: its ring (shared address, 1024-aligned), the NS
// full barriers, a generic pointer to the ring (the epilogue's scratch sits
// in it: the stages are free by then), the quantized pools' scale array
// (shared address and generic pointer), and the blocks consumed so far.
struct WarpPipe {
    uint32_t ring;
    uint32_t bars;
    uint8_t *stage_ptr;
    uint32_t scales;
    const float *scale_f;
    uint32_t seq;
};

// Decode item `item` of list dl: items of listed request li are
// dl.item_off[li] .. dl.item_off[li + 1] - 1, split-major with the KV heads
// adjacent (item = item_off + split * hkv + kh).  Unsplit requests write
// bf16 rows; split ones write fp32 partials (o, m, l) at rows
// part_off + (split * t + i) * hq + h and count on their counter (cnt_off +
// kh): the warp that counts last merges the splits.  Combined calls (fw_k):
// the item whose key range holds the request's new rows writes them into the
// pool first.
template <int DP, int D, int NS, bool FP8 = false>
__device__ __forceinline__ void warp_decode_item(const AttnParams &p, const WorkList &dl, int item, WarpPipe &wp,
                                                 const DecodeMaps &maps)
{
    static_assert(!FP8 || (DP == 128 && D == 128), "quantized pools have head dim 128");
    constexpr int kSlice = FP8 ? WarpRingF8::kSlice : WarpRing<DP>::kSlice;
    constexpr int kStage = FP8 ? WarpRingF8::kStage : WarpRing<DP>::kStage;
    constexpr int kTx = FP8 ? WarpRingF8::kBytes : WarpRing<DP>::kBytes;
    const int lane = threadIdx.x & 31;
    const int li = find_listed(dl, item);
    const int local = item - dl.item_off[li];
    const int split = local / p.hkv, kh = local - split * p.hkv;
    const int r = dl.req[li];
    const int b = dl.qb[li], t = dl.qt[li], L = dl.len[li];
    const int g = p.group;
    const int nr = t * g;
    if (L == 0 || t == 0) {                                        // padding request: zero rows
        if (split == 0) {
            if (p.fw_k && t > 0) {
                if constexpr (!FP8) fused_kv_write<D>(p, r, b, t, 0, kh, -t, 0, lane, 32);
                else fused_kv_write_fp8(p, r, b, t, 0, kh, 1, -t, 0, lane);
            }
            for (int idx = lane; idx < nr * D; idx += 32) {
                const int rr = idx / D, e = idx - rr * D;
                p.out[((size_t)(b + rr / g) * p.hq + kh * g + rr % g) * D + e] = __float2bfloat16(0.f);
            }
            if (kh == 0 && lane == 0) check_meta(p, dl, li);
        }
        return;
    }
    const int k_begin = decode_key_begin(t, L, p.window) + split * dl.split_tokens;
    const int k_end = min(L, k_begin + dl.split_tokens);
    const bool partial = dl.part_off[li] >= 0;
    const int blk0 = k_begin >> 4;
    const int nblk = ((k_end + 15) >> 4) - blk0;
    const int32_t *bt = p.block_table + (size_t)r * p.bt_stride + blk0;
    int ids = lane < nblk ? __ldg(bt + lane) : 0;
    if (p.fw_k) {                                                  // combined call: this item's new rows first
        if constexpr (!FP8) fused_kv_write<D>(p, r, b, t, L, kh, max(k_begin, L - t), min(k_end, L), lane, 32);
        else fused_kv_write_fp8(p, r, b, t, L, kh, 1, max(k_begin, L - t), min(k_end, L), lane);
        __syncwarp();
        fence_proxy_async_global();
    }
    auto issue = [&](int j) {                                      // block j of the item (every lane; ids current)
        int blk = __shfl_sync(0xffffffffu, ids, j & 31);
        if (blk < 0 || blk >= p.nb_total) {                        // outside the pool: report, read block 0
            if (lane == 0) atomicOr(p.err, 2u);
            blk = 0;
        }
        const int s = (wp.seq + j) % NS;
        const uint32_t st = wp.ring + s * kStage, bar = wp.bars + 8u * s;
        if constexpr (FP8) {
            // lane i < 16: the K scale of the block's slot i, lane 16 + i its
            // V scale; every lane's arrival is counted before lane 0's
            const int key = lane & 15;
            const float *src = (lane < 16 ? p.k_scale : p.v_scale) + ((int64_t)blk * 16 + key) * p.hkv + kh;
            cp_async_4(wp.scales + s * WarpRingF8::kScaleStage + lane * 4, src);
            cp_async_mbar_arrive(bar);
            __syncwarp();
        }
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, kTx);
            if constexpr (FP8) {
                tma_load_3d(st, &maps.k, bar, 0, kh, blk * 16);
                tma_load_3d(st + kSlice, &maps.v, bar, 0, kh, blk * 16);
            } else {
#pragma unroll
                for (int x = 0; x < DP / 64; x++) {
                    tma_load_3d(st + x * 2048, &maps.k, bar, x * 64, kh, blk * 16);
                    tma_load_3d(st + kSlice + x * 2048, &maps.v, bar, x * 64, kh, blk * 16);
                }
            }
        }
    };
    const int pre = nblk < NS ? nblk : NS;
    for (int j = 0; j < pre; j++) issue(j);

    const int rq = lane >> 2, c2 = 2 * (lane & 3);
    const int mi = lane >> 3, mr = lane & 7;
    uint32_t qb[DP / 16][2];
    const size_t qrow = rq < nr ? (size_t)(b + rq / g) * p.hq + kh * g + rq % g : 0;
    if constexpr (FP8) load_qt_frags<D, true>(qb, p.q, qrow, rq < nr, lane);
    else load_qt_frags_pad<DP, D>(qb, p.q, qrow, rq < nr, lane);
    const int qbase = L - t;
    const int qp0 = c2 < nr ? qbase + c2 / g : -1;
    const int qp1 = c2 + 1 < nr ? qbase + (c2 + 1) / g : -1;
    const int wspan = win_span(p.window);
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    float o[DP / 16][4];
#pragma unroll
    for (int n = 0; n < DP / 16; n++) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    bool alive = true;
    int consumed = 0, issued = pre;
    for (int j = 0; j < nblk; j++) {
        const int s = (wp.seq + j) % NS;
        if (!__all_sync(0xffffffffu, mbar_wait(wp.bars + 8u * s, ((wp.seq + j) / NS) & 1, p.err))) {
            alive = false;
            break;
        }
        consumed = j + 1;
        const uint32_t kt = wp.ring + s * kStage;
        float sc[1][4] = {{0.f, 0.f, 0.f, 0.f}}, vs[1][2] = {{1.f, 1.f}};
        const uint32_t vt[1] = {kt + kSlice};
        const bool has[1] = {true};
        block_scores_t<DP, FP8>(sc[0], qb, kt, mi, mr);
        float f0 = p.scale_log2, f1 = p.scale_log2;
        if constexpr (FP8) {                                       // K and V scales of keys rq, rq + 8
            const float *sk = wp.scale_f + s * (WarpRingF8::kScaleStage / 4);
            f0 *= sk[rq];
            f1 *= sk[rq + 8];
            vs[0][0] = sk[16 + rq];
            vs[0][1] = sk[16 + rq + 8];
        }
        mask_scale_t(sc[0], ((blk0 + j) << 4) + rq, k_end, qp0, qp1, wspan, true, f0, f1);
        softmax_pv_t<DP, FP8, 1>(o, m, l, sc, vs, vt, has, mi, mr);
        __syncwarp();
        if (j + NS < nblk) {
            // the slot's reads are done; make them precede the copy that refills it
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            if (((j + NS) & 31) == 0) ids = j + NS + lane < nblk ? __ldg(bt + j + NS + lane) : 0;
            issue(j + NS);
            issued = j + NS + 1;
        }
    }
    if (!alive && lane == 0) {                                     // drain this warp's copies still in flight
        for (int j = consumed; j < issued; j++) mbar_wait(wp.bars + 8u * ((wp.seq + j) % NS), ((wp.seq + j) / NS) & 1, p.err);
    }
    __syncwarp();
    wp.seq += issued;

    // ---- epilogue: rows through the (now free) ring memory
#pragma unroll
    for (int j = 0; j < 2; j++) {
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 4);
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 8);
        l[j] += __shfl_xor_sync(0xffffffffu, l[j], 16);
    }
    float *mo = reinterpret_cast<float *>(wp.stage_ptr);          // [8][DP] then (m, l) [8][2]
    float *mml = mo + 8 * DP;
#pragma unroll
    for (int j = 0; j < 2; j++) {
        const int x = c2 + j;
#pragma unroll
        for (int mt = 0; mt < DP / 16; mt++) {
            mo[x * DP + ot_dim<FP8>(mt, rq, 0)] = o[mt][j];
            mo[x * DP + ot_dim<FP8>(mt, rq, 1)] = o[mt][2 + j];
        }
        if (rq == 0) {
            mml[x * 2] = m[j];
            mml[x * 2 + 1] = l[j];
        }
    }
    __syncwarp();
    constexpr int kChunks = D / 8;
    for (int idx = lane; alive && idx < nr * kChunks; idx += 32) {
        const int rr = idx / kChunks, e0 = (idx - rr * kChunks) * 8;
        const int i = rr / g, h = kh * g + rr % g;
        const float *src = mo + rr * DP + e0;
        if (!partial) {
            const float ls = mml[rr * 2 + 1];
            const float inv = ls > 0.f ? 1.f / ls : 0.f;
            uint4 v;
            v.x = pack_bf16x2(src[0] * inv, src[1] * inv);
            v.y = pack_bf16x2(src[2] * inv, src[3] * inv);
            v.z = pack_bf16x2(src[4] * inv, src[5] * inv);
            v.w = pack_bf16x2(src[6] * inv, src[7] * inv);
            *reinterpret_cast<uint4 *>(p.out + ((size_t)(b + i) * p.hq + h) * D + e0) = v;
        } else {
            const size_t orow = (size_t)dl.part_off[li] + ((size_t)split * t + i) * p.hq + h;
            float4 *dst = reinterpret_cast<float4 *>(p.part_o + orow * D + e0);
            dst[0] = make_float4(src[0], src[1], src[2], src[3]);
            dst[1] = make_float4(src[4], src[5], src[6], src[7]);
            if (e0 == 0) p.part_ml[orow] = make_float2(mml[rr * 2], mml[rr * 2 + 1]);
        }
    }
    if (kh == 0 && split == 0 && lane == 0) check_meta(p, dl, li);
    __syncwarp();
    if (!partial) return;
    // ---- split request: count this split; the warp counting last merges them
    const int S = decode_splits(t, L, p.window, dl.split_tokens);
    uint32_t *cnt = p.counters + (size_t)(dl.cnt_off[li] + kh) * kCounterStride;
    uint32_t last = 0u;
    if (lane == 0) {
        __threadfence();                                           // release this split's partials
        const uint32_t old = atomicAdd(cnt, 1u);
        if (old >= (uint32_t)S) atomicOr(p.err, kDevErrCounter);  // the workspace was not zero-filled
        last = old + 1u == (uint32_t)S ? 1u : 0u;
        if (last) __threadfence();                                 // acquire the other splits' partials
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    if (!last) return;
    combine_in_cta<D>(p, (size_t)dl.part_off[li], b, t, kh, g, S, lane, 32);
    __syncwarp();
    if (lane == 0) atomicExch(cnt, 0u);                            // ready for the next call
}

}  // namespace pkv

// Ragged paged attention for prefill chunks on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), head_dim 128.
//
// One CTA = (listed request, KV head, tile of 128 query rows).  A row is a
// (token, query head) pair of the KV head's group: 128/g consecutive new
// tokens x g heads (the vllm-lite README's grouped-query fold, so a K/V tile
// feeds all g heads in one MMA).  Query i of a request with t new tokens and
// context L sits at position L - t + i and sees keys 0 .. that position
// ("31. Engine v2", "Attention over the pool").  Keys are taken in tiles of
// 128 = 8 paged blocks, each block's 16-row K and V slices of this KV head
// copied by TMA straight from the pool through the block table (key j lives
// in block table[j / 16], row j % 16): the paged layout is read in place.
//
// Warp roles (256 threads):
//   warp 0      TMA producer: Q once, then K and V tiles into a 2-stage ring;
//   warp 1      MMA issuer (one thread): S = Q K^T into a double-buffered
//               TMEM tile, then O += P V into a TMEM accumulator;
//   warps 4..7  softmax, one thread per row (TMEM lane): S row from TMEM,
//               causal mask, online softmax in the exp2 domain with the
//               running max only moved (and O rescaled in TMEM) when it
//               grows by more than 2^8, P written to shared memory in the
//               MMA's operand layout; at the end O / l to bf16 output.
// The MMA for S(j+1) runs while the softmax works on S(j).
//
// All shared-memory operands use the 128-byte swizzle: Q, K and P are
// K-major ([rows][64 columns] sub-tiles), V is MN-major ([keys][64 dims]).
#include <climits>
#include <mutex>

#include "common.cuh"
#include "sm100.cuh"

namespace pkv {

constexpr int kTcThreads = 256;
constexpr int kTcRows = 128;          // query rows per CTA (MMA M)
constexpr int kTcKeys = 128;          // keys per tile (MMA N of S, K of PV)
constexpr int kTcD = 128;
constexpr int kSub = 16384;           // one [128][64] bf16 sub-tile
constexpr int kTile = 2 * kSub;       // [128][128]
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kTile;                  // 2 stages
constexpr int kVOff = kKOff + 2 * kTile;              // 2 stages
constexpr int kPOff = kVOff + 2 * kTile;
constexpr int kBarOff = kPOff + kTile;
constexpr int kTcSmem = 1024 + kBarOff + 256;
constexpr uint32_t kTmemCols = 512;   // S0 [0,128), S1 [128,256), O [256,384)
constexpr float kRescaleLog2 = 8.0f;  // move the running max only when it grows by more than this

enum TcBar {
    kBarQ = 0,
    kBarK0 = 1, kBarK1 = 2,
    kBarV0 = 3, kBarV1 = 4,
    kBarKVEmpty0 = 5, kBarKVEmpty1 = 6,
    kBarS0 = 7, kBarS1 = 8,
    kBarSFree0 = 9, kBarSFree1 = 10,
    kBarP = 11,
    kBarO = 12,
    kBarMmaDone = 13,
    kNumTcBars = 14
};

// byte offset of 16-byte chunk c (8 columns) of row `row` in a [128][128]
// K-major tile made of two swizzled [128][64] sub-tiles
__device__ __forceinline__ uint32_t kmaj_off(int row, int c)
{
    return (c >> 3) * kSub + (row >> 3) * 1024 + (row & 7) * 128 + (((c & 7) ^ (row & 7)) << 4);
}

__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(AttnParams p, const __grid_constant__ WorkList wl,
                                                                const __grid_constant__ CUtensorMap qmap,
                                                                const __grid_constant__ CUtensorMap kmap,
                                                                const __grid_constant__ CUtensorMap vmap,
                                                                int64_t num_slots)
{
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sb = (raw + 1023u) & ~1023u;
    uint8_t *sp = smem_raw + (sb - raw);
    auto bar = [&](int i) { return sb + kBarOff + 8u * i; };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sp + kBarOff + 8 * kNumTcBars);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int kh = blockIdx.y;
    const int li = find_listed(wl, blockIdx.x);
    const int r = wl.req[li];
    const int b = p.qsl[r], t = p.qsl[r + 1] - b, L = p.seq_lens[r];
    const int g = p.group;
    const int tile_tokens = wl.tile_tokens;                       // 128 / g
    const int ntiles = (t + tile_tokens - 1) / tile_tokens;
    const int tile = ntiles - 1 - (blockIdx.x - wl.item_off[li]);   // longest tiles first
    const int i0 = tile * tile_tokens;
    const int ntok = min(tile_tokens, t - i0);
    const int nr = ntok * g;
    const int k_end = L - t + i0 + ntok;                           // one past the last position
    const int nkt = (k_end + kTcKeys - 1) / kTcKeys;               // key tiles
    const int nblk = (k_end + 15) >> 4;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kNumTcBars; i++) {
            uint32_t cnt = 1;
            if (i == kBarSFree0 || i == kBarSFree1 || i == kBarP) cnt = 4;
            mbar_init(bar(i), cnt);
        }
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

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tmap(&qmap);
            prefetch_tmap(&kmap);
            prefetch_tmap(&vmap);
            mbar_arrive_expect_tx(bar(kBarQ), kTile);
            tma_load_3d(sb + kQOff, &qmap, bar(kBarQ), 0, kh * g, b + i0);
            tma_load_3d(sb + kQOff + kSub, &qmap, bar(kBarQ), 64, kh * g, b + i0);
        }
        const int32_t *bt = p.block_table + (size_t)r * p.bt_stride;
        int ids = 0, issued = 0;
        for (int j = 0; j < nkt; j++) {
            const int st = j & 1;
            if ((j & 3) == 0) {                                    // 32 block ids = 4 key tiles
                const int jb = j * 8 + lane;
                ids = jb < nblk ? __ldg(bt + jb) : INT_MIN;
            }
            bool ok = true;
            if (j >= 2) ok = mbar_wait(bar(kBarKVEmpty0 + st), ((j >> 1) - 1) & 1, p.err);
            if (!__all_sync(0xffffffffu, ok)) break;
            issued = j + 1;
            if (lane == 0) {
                mbar_arrive_expect_tx(bar(kBarK0 + st), kTile);
                mbar_arrive_expect_tx(bar(kBarV0 + st), kTile);
            }
            for (int bi = 0; bi < 8; bi++) {
                int blk = __shfl_sync(0xffffffffu, ids, ((j & 3) << 3) + bi);
                if (lane == 0) {
                    int row = (int)num_slots;                      // beyond the pool: TMA fills zeros
                    if (blk != INT_MIN) {                          // a block of the key range
                        if (blk < 0 || blk >= p.nb_total) atomicOr(p.err, 2u);
                        else row = blk * 16;
                    }
                    const uint32_t kd = sb + kKOff + st * kTile + bi * 2048;
                    const uint32_t vd = sb + kVOff + st * kTile + bi * 2048;
                    tma_load_3d(kd, &kmap, bar(kBarK0 + st), 0, kh, row);
                    tma_load_3d(kd + kSub, &kmap, bar(kBarK0 + st), 64, kh, row);
                    tma_load_3d(vd, &vmap, bar(kBarV0 + st), 0, kh, row);
                    tma_load_3d(vd + kSub, &vmap, bar(kBarV0 + st), 64, kh, row);
                }
            }
            __syncwarp();
        }
        if (issued < nkt && lane == 0) {                           // a wait gave up: drain own copies
            for (int j = issued > 2 ? issued - 2 : 0; j < issued; j++) {
                mbar_wait(bar(kBarK0 + (j & 1)), (j >> 1) & 1, p.err);
                mbar_wait(bar(kBarV0 + (j & 1)), (j >> 1) & 1, p.err);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16(kTcRows, kTcKeys, false);
            constexpr uint32_t idO = idesc_bf16(kTcRows, kTcD, true);
            bool ok = mbar_wait(bar(kBarQ), 0, p.err);
            auto issue_pv = [&](int i) -> bool {
                if (!mbar_wait(bar(kBarP), i & 1, p.err)) return false;
                if (!mbar_wait(bar(kBarV0 + (i & 1)), (i >> 1) & 1, p.err)) return false;
                tc_fence_after();
                const uint32_t vbase = sb + kVOff + (i & 1) * kTile;
#pragma unroll
                for (int kk = 0; kk < 8; kk++) {
                    const uint64_t ad = sdesc_sw128(sb + kPOff + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(vbase + kk * 2048, kSub, 1024);
                    tc_mma(tmem + 256, ad, bd, idO, (i > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar(kBarO));
                tc_commit(bar(kBarKVEmpty0 + (i & 1)));
                return true;
            };
            for (int j = 0; j < nkt && ok; j++) {
                const int s = j & 1;
                ok = mbar_wait(bar(kBarK0 + s), (j >> 1) & 1, p.err);
                if (ok && j >= 2) ok = mbar_wait(bar(kBarSFree0 + s), ((j >> 1) - 1) & 1, p.err);
                if (!ok) break;
                tc_fence_after();
                const uint32_t kbase = sb + kKOff + s * kTile;
#pragma unroll
                for (int kk = 0; kk < 8; kk++) {
                    const uint64_t ad = sdesc_sw128(sb + kQOff + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = sdesc_sw128(kbase + (kk >> 2) * kSub + (kk & 3) * 32, 16, 1024);
                    tc_mma(tmem + s * 128, ad, bd, idS, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(kBarS0 + s));
                if (j >= 1) ok = issue_pv(j - 1);
            }
            if (ok) issue_pv(nkt - 1);
            // every MMA this thread issued has finished before TMEM is released
            tc_commit(bar(kBarMmaDone));
            mbar_wait(bar(kBarMmaDone), 0, p.err);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax, one row per thread
        const int row = threadIdx.x - 128;
        const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const int qpos = row < nr ? L - t + i0 + row / g : -1;
        const float sl2 = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < nkt; j++) {
            const int s = j & 1;
            ok = mbar_wait(bar(kBarS0 + s), (j >> 1) & 1, p.err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc_fence_after();
            float x[kTcKeys];
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t v[32];
                tmem_ld32(tl + s * 128 + c * 32, v);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 32; k++) x[c * 32 + k] = __uint_as_float(v[k]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarSFree0 + s));

            const int key0 = j * kTcKeys;
            float mt = -INFINITY;
            if (key0 + kTcKeys - 1 <= qpos) {
#pragma unroll
                for (int k = 0; k < kTcKeys; k++) {
                    x[k] *= sl2;
                    mt = fmaxf(mt, x[k]);
                }
            } else {
#pragma unroll
                for (int k = 0; k < kTcKeys; k++) {
                    x[k] = (key0 + k <= qpos) ? x[k] * sl2 : -INFINITY;
                    mt = fmaxf(mt, x[k]);
                }
            }
            if (j > 0) {
                // PV(j-1) has finished: O is stable and the P buffer is free
                ok = mbar_wait(bar(kBarO), (j - 1) & 1, p.err);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                tc_fence_after();
                const bool need = mt > m_used + kRescaleLog2;
                if (__any_sync(0xffffffffu, need)) {
                    const float alpha = need ? exp2f(m_used - mt) : 1.f;
                    if (need) {
                        l *= alpha;
                        m_used = mt;
                    }
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        uint32_t v[32];
                        tmem_ld32(tl + 256 + c * 32, v);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; k++) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
                        tmem_st32(tl + 256 + c * 32, v);
                    }
                    tmem_st_wait();
                }
            } else {
                m_used = mt;
            }
            const float ms = m_used == -INFINITY ? 0.f : m_used;
            uint8_t *prow = sp + kPOff;
#pragma unroll
            for (int c = 0; c < 16; c++) {
                uint32_t w4[4];
#pragma unroll
                for (int q = 0; q < 4; q++) {
                    const float p0 = exp2f(x[c * 8 + 2 * q] - ms);
                    const float p1 = exp2f(x[c * 8 + 2 * q + 1] - ms);
                    l += p0 + p1;
                    w4[q] = pack_bf16x2(p0, p1);
                }
                *reinterpret_cast<uint4 *>(prow + kmaj_off(row, c)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarP));
        }
        if (ok) ok = mbar_wait(bar(kBarO), (nkt - 1) & 1, p.err);
        if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const size_t orow = row < nr ? ((size_t)(b + i0 + row / g) * p.hq + kh * g + row % g) * kTcD : 0;
#pragma unroll
            for (int c = 0; c < 4; c++) {
                uint32_t v[32];
                tmem_ld32(tl + 256 + c * 32, v);
                tmem_ld_wait();
                if (row < nr) {
                    uint4 *dst = reinterpret_cast<uint4 *>(p.out + orow + c * 32);
#pragma unroll
                    for (int q = 0; q < 4; q++) {
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
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

cudaError_t make_pool_tmap(CUtensorMap *map, const void *pool, int64_t num_slots, int hkv, int d, int box_cols,
                           bool swizzle128);
cudaError_t make_q_tmap(CUtensorMap *map, const void *q, int num_tokens, int hq, int d, int g);

bool tc_prefill_supported(int head_dim, int group) { return head_dim == kTcD && group >= 1 && kTcRows % group == 0; }
int tc_prefill_rows() { return kTcRows; }

cudaError_t launch_attn_tc(const AttnParams &p, const WorkList &wl, int num_items, const void *q, int num_tokens,
                           const void *k_cache, const void *v_cache, int64_t num_slots, cudaStream_t stream)
{
    if (num_items <= 0) return cudaSuccess;
    static std::once_flag once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(once, [] {
        attr_err = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem);
    });
    if (attr_err != cudaSuccess) return attr_err;
    CUtensorMap qm, km, vm;
    cudaError_t e = make_q_tmap(&qm, q, num_tokens, p.hq, kTcD, p.group);
    if (e == cudaSuccess) e = make_pool_tmap(&km, k_cache, num_slots, p.hkv, kTcD, 64, true);
    if (e == cudaSuccess) e = make_pool_tmap(&vm, v_cache, num_slots, p.hkv, kTcD, 64, true);
    if (e != cudaSuccess) return e;
    dim3 grid(num_items, p.hkv);
    launch_begin(stream, kAttnTcPrefill);
    attn_tc_kernel<<<grid, kTcThreads, kTcSmem, stream>>>(p, wl, qm, km, vm, num_slots);
    launch_end(stream);
    return cudaGetLastError();
}

}  // namespace pkv

// Ragged paged attention on CUDA cores (fp32 FMA).
//
// One CTA = (listed request, KV head, item).  An item is a KV split of a
// decode-class request (all of its t <= 16/g new tokens, keys
// [s*split, (s+1)*split)) or a tile of a prefill-class request's new tokens
// (keys 0 .. the tile's last position).  The rows of a CTA are the
// (token, query head) pairs that share KV head kh: the vllm-lite README's
// grouped-query fold (query heads of a group read one KV head, never a
// repeated copy), so every K/V row is loaded once for all g heads.
//
// Keys are gathered through the block table ("31. Engine v2", "Attention
// over the pool": key position j lives in block table[j / 16] at row
// j % 16).  Query i of a request with t new tokens and context L sits at
// position L - t + i and sees keys 0 .. that position.  Softmax is the
// online (running max / running sum) form of exact attention, in the exp2
// domain with scale*log2(e) folded into q; each of the 4 warps keeps its
// own state over a strided quarter of the keys and the warps merge at the
// end.  Unsplit items write bf16 output; split items write fp32 partials
// (unnormalised o, running max, weight sum) for the combine kernel.
#include "common.cuh"
#include "sm100.cuh"

namespace pkv {

constexpr int kFmaThreads = 128;
constexpr int kFmaWarps = kFmaThreads / 32;
constexpr int kBlock = 16;                       // tokens per KV block

template <int D>
struct FmaShape {
    static constexpr int EPL = D >= 128 ? 4 : 2;           // V elements per lane
    static constexpr int NCH = D / 8;                      // 16-byte chunks per K row
};

template <int D, int R>
__host__ __device__ constexpr int fma_smem_floats()
{
    return (R * D + kFmaWarps * R * 32) > (kFmaWarps * R * D + 2 * kFmaWarps * R)
               ? (R * D + kFmaWarps * R * 32)
               : (kFmaWarps * R * D + 2 * kFmaWarps * R);
}

template <int D, int R>
__global__ void __launch_bounds__(kFmaThreads) attn_fma_kernel(AttnParams p,
                                                               const __grid_constant__ WorkList wl)
{
    constexpr int EPL = FmaShape<D>::EPL;
    constexpr int NCH = FmaShape<D>::NCH;
    extern __shared__ float4 smem_f4[];
    float *q_s = reinterpret_cast<float *>(smem_f4);              // [R][D] q * scale*log2e
    float *p_s = q_s + R * D;                                     // [warps][R][32] weights
    float *mo_s = q_s;                                            // after the loop: [warps][R][D]
    float *mm_s = mo_s + kFmaWarps * R * D;                       // [warps][R]
    float *ml_s = mm_s + kFmaWarps * R;                           // [warps][R]

    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int kh = blockIdx.y;
    const int li = find_listed(wl, blockIdx.x);
    const int local = blockIdx.x - wl.item_off[li];
    const int r = wl.req[li];
    const int b = wl.qb[li], t = wl.qt[li], L = wl.len[li];
    const int g = p.group;
    if (tid == 0 && local == 0 && kh == 0) check_meta(p, wl, li);

    if (L == 0 || t == 0) {                       // padding request: its rows are zero
        for (int idx = tid; idx < t * g * D; idx += kFmaThreads) {
            int rr = idx / D, e = idx - rr * D;
            int i = rr / g, h = kh * g + rr % g;
            p.out[((size_t)(b + i) * p.hq + h) * D + e] = __float2bfloat16(0.f);
        }
        return;
    }

    int i0, nt, k_begin, k_end, split = 0;
    bool partial = false;
    if (wl.mode == kModeDecode) {
        i0 = 0;
        nt = t;
        split = local;
        k_begin = decode_key_begin(t, L, p.window) + split * wl.split_tokens;
        k_end = min(L, k_begin + wl.split_tokens);
        partial = wl.part_off[li] >= 0;
    } else {
        i0 = local * wl.tile_tokens;
        nt = min(wl.tile_tokens, t - i0);
        k_begin = window_lo(L - t + i0, p.window) & ~15;  // the first row's window start
        k_end = L - t + i0 + nt;                  // one past the tile's last query position
    }
    const int wspan = win_span(p.window);         // keys <= position - wspan are outside the window
    const int nr = nt * g;

    for (int idx = tid; idx < R * D; idx += kFmaThreads) {
        int rr = idx / D, e = idx - rr * D;
        float val = 0.f;
        if (rr < nr) {
            int i = i0 + rr / g, h = kh * g + rr % g;
            val = __bfloat162float(p.q[((size_t)(b + i) * p.hq + h) * D + e]) * p.scale_log2;
        }
        q_s[idx] = val;
    }

    int qpos[R];
#pragma unroll
    for (int rr = 0; rr < R; rr++) qpos[rr] = (rr < nr) ? L - t + i0 + rr / g : -1;

    float m[R], l[R], o[R][EPL];
#pragma unroll
    for (int rr = 0; rr < R; rr++) {
        m[rr] = -INFINITY;
        l[rr] = 0.f;
#pragma unroll
        for (int x = 0; x < EPL; x++) o[rr][x] = 0.f;
    }
    __syncthreads();

    const int32_t *bt = p.block_table + (size_t)r * p.bt_stride;
    const size_t slot_elems = (size_t)p.hkv * D;
    float *pw = p_s + w * R * 32;
    const bool v_lane = lane * EPL < D;

    for (int kb = k_begin + w * 32; kb < k_end; kb += kFmaWarps * 32) {
        const int j = kb + lane;
        bool valid = j < k_end;
        int blk = 0, row = 0;
        if (valid) {
            blk = __ldg(bt + j / kBlock);
            row = j % kBlock;
            if (blk < 0 || blk >= p.nb_total) {   // outside the pool: report, read nothing
                atomicOr(p.err, 2u);
                valid = false;
                blk = 0;
                row = 0;
            }
        }
        const size_t base = ((size_t)blk * kBlock + row) * slot_elems + (size_t)kh * D;

        float s[R];
#pragma unroll
        for (int rr = 0; rr < R; rr++) s[rr] = 0.f;
        const uint4 *krow = reinterpret_cast<const uint4 *>(p.k_cache + base);
#pragma unroll
        for (int c = 0; c < NCH; c++) {
            const uint4 kv = ldg_nc_v4(krow + c);
            const float kf[8] = {bf16_lo(kv.x), bf16_hi(kv.x), bf16_lo(kv.y), bf16_hi(kv.y),
                                 bf16_lo(kv.z), bf16_hi(kv.z), bf16_lo(kv.w), bf16_hi(kv.w)};
#pragma unroll
            for (int rr = 0; rr < R; rr++) {
                const float4 qa = *reinterpret_cast<const float4 *>(q_s + rr * D + c * 8);
                const float4 qb = *reinterpret_cast<const float4 *>(q_s + rr * D + c * 8 + 4);
                float a = s[rr];
                a = fmaf(qa.x, kf[0], a);
                a = fmaf(qa.y, kf[1], a);
                a = fmaf(qa.z, kf[2], a);
                a = fmaf(qa.w, kf[3], a);
                a = fmaf(qb.x, kf[4], a);
                a = fmaf(qb.y, kf[5], a);
                a = fmaf(qb.z, kf[6], a);
                a = fmaf(qb.w, kf[7], a);
                s[rr] = a;
            }
        }

        float alpha[R];
#pragma unroll
        for (int rr = 0; rr < R; rr++) {
            const float sv = (valid && j <= qpos[rr] && j > qpos[rr] - wspan) ? s[rr] : -INFINITY;
            const float mnew = fmaxf(m[rr], warp_max(sv));
            const float msafe = mnew == -INFINITY ? 0.f : mnew;
            alpha[rr] = exp2f(m[rr] - msafe);
            const float pv = exp2f(sv - msafe);
            l[rr] = l[rr] * alpha[rr] + pv;
            m[rr] = mnew;
            pw[rr * 32 + lane] = pv;
        }
        __syncwarp();

#pragma unroll
        for (int rr = 0; rr < R; rr++)
#pragma unroll
            for (int x = 0; x < EPL; x++) o[rr][x] *= alpha[rr];

        const int nkeys = min(32, k_end - kb);
        for (int jj = 0; jj < nkeys; jj += 4) {
            float vf[4][EPL];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const size_t bu = __shfl_sync(0xffffffffu, (unsigned long long)base, jj + u);
                if (v_lane) {
                    const __nv_bfloat16 *vp = p.v_cache + bu + lane * EPL;
                    if constexpr (EPL == 4) {
                        const uint2 vv = __ldg(reinterpret_cast<const uint2 *>(vp));
                        vf[u][0] = bf16_lo(vv.x);
                        vf[u][1] = bf16_hi(vv.x);
                        vf[u][2] = bf16_lo(vv.y);
                        vf[u][3] = bf16_hi(vv.y);
                    } else {
                        const uint32_t vv = __ldg(reinterpret_cast<const uint32_t *>(vp));
                        vf[u][0] = bf16_lo(vv);
                        vf[u][1] = bf16_hi(vv);
                    }
                } else {
#pragma unroll
                    for (int x = 0; x < EPL; x++) vf[u][x] = 0.f;
                }
            }
#pragma unroll
            for (int rr = 0; rr < R; rr++) {
                const float4 pp = *reinterpret_cast<const float4 *>(pw + rr * 32 + jj);
#pragma unroll
                for (int x = 0; x < EPL; x++) {
                    float a = o[rr][x];
                    a = fmaf(pp.x, vf[0][x], a);
                    a = fmaf(pp.y, vf[1][x], a);
                    a = fmaf(pp.z, vf[2][x], a);
                    a = fmaf(pp.w, vf[3][x], a);
                    o[rr][x] = a;
                }
            }
        }
        __syncwarp();
    }

#pragma unroll
    for (int rr = 0; rr < R; rr++) l[rr] = warp_sum(l[rr]);
    __syncthreads();                                          // q_s / p_s are dead from here
    if (v_lane) {
#pragma unroll
        for (int rr = 0; rr < R; rr++)
#pragma unroll
            for (int x = 0; x < EPL; x++) mo_s[(w * R + rr) * D + lane * EPL + x] = o[rr][x];
    }
    if (lane == 0) {
#pragma unroll
        for (int rr = 0; rr < R; rr++) {
            mm_s[w * R + rr] = m[rr];
            ml_s[w * R + rr] = l[rr];
        }
    }
    __syncthreads();

    for (int idx = tid; idx < nr * D; idx += kFmaThreads) {
        const int rr = idx / D, e = idx - rr * D;
        float M = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < kFmaWarps; ww++) M = fmaxf(M, mm_s[ww * R + rr]);
        const float Ms = M == -INFINITY ? 0.f : M;
        float acc = 0.f, ls = 0.f;
#pragma unroll
        for (int ww = 0; ww < kFmaWarps; ww++) {
            const float sc = exp2f(mm_s[ww * R + rr] - Ms);
            acc = fmaf(sc, mo_s[(ww * R + rr) * D + e], acc);
            ls = fmaf(sc, ml_s[ww * R + rr], ls);
        }
        const int i = i0 + rr / g, h = kh * g + rr % g;
        if (!partial) {
            p.out[((size_t)(b + i) * p.hq + h) * D + e] = __float2bfloat16(ls > 0.f ? acc / ls : 0.f);
        } else {
            const size_t prow = (size_t)wl.part_off[li] + ((size_t)split * t + i) * p.hq + h;
            p.part_o[prow * D + e] = acc;
            if (e == 0) p.part_ml[prow] = make_float2(M, ls);
        }
    }
}

template <int D, int R>
static cudaError_t launch_fma_dr(const AttnParams &p, const WorkList &wl, int num_items,
                                 cudaStream_t stream)
{
    constexpr int smem = fma_smem_floats<D, R>() * 4;
    static_assert(smem <= 48 * 1024, "FMA attention smem above the default limit");
    dim3 grid(num_items, p.hkv);
    launch_begin(stream, wl.mode == kModeDecode ? kAttnFmaDecode : kAttnFmaPrefill);
    attn_fma_kernel<D, R><<<grid, kFmaThreads, smem, stream>>>(p, wl);
    launch_end(stream);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_fma_d(const AttnParams &p, const WorkList &wl, int rows, int num_items,
                                cudaStream_t stream)
{
    if (rows <= 4) return launch_fma_dr<D, 4>(p, wl, num_items, stream);
    if (rows <= 8) return launch_fma_dr<D, 8>(p, wl, num_items, stream);
    return launch_fma_dr<D, 16>(p, wl, num_items, stream);
}

cudaError_t launch_attn_fma(const AttnParams &p, const WorkList &wl, int head_dim, int rows,
                            int num_items, cudaStream_t stream)
{
    if (num_items <= 0) return cudaSuccess;
    switch (head_dim) {
    case 48: return launch_fma_d<48>(p, wl, rows, num_items, stream);
    case 64: return launch_fma_d<64>(p, wl, rows, num_items, stream);
    case 128: return launch_fma_d<128>(p, wl, rows, num_items, stream);
    default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------- split-KV combine
//
// Row (token i, head h) of a split request r has partials from
// S = ceil(L / split) splits: o_s (unnormalised), m_s (running max, exp2
// domain) and l_s (weight sum).  The exact result is
//   o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,   M = max_s m_s.
// One warp per row, lanes across head_dim.
template <int D>
__global__ void __launch_bounds__(256) attn_combine_kernel(AttnParams p,
                                                           const __grid_constant__ WorkList wl)
{
    constexpr int EPL = FmaShape<D>::EPL;
    const int li = blockIdx.x;
    const int b = wl.qb[li], t = wl.qt[li], L = wl.len[li];
    // decode-class requests split their (windowed) key range; every tile of a
    // split prefill request has ceil(L / split) splits
    const int S = wl.mode == kModeDecode ? decode_splits(t, L, p.window, wl.split_tokens)
                                         : (L + wl.split_tokens - 1) / wl.split_tokens;
    const int rows = t * p.hq;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.y * (blockDim.x / 32) + (threadIdx.x >> 5);
    pdl_wait();                                                   // the split partials are written
    if (row >= rows) return;
    const size_t base = (size_t)wl.part_off[li];

    float M = -INFINITY;
    for (int s = lane; s < S; s += 32) M = fmaxf(M, p.part_ml[base + (size_t)s * rows + row].x);
    M = warp_max(M);
    const float Ms = M == -INFINITY ? 0.f : M;
    float acc[EPL], ls = 0.f;
#pragma unroll
    for (int x = 0; x < EPL; x++) acc[x] = 0.f;
    const bool v_lane = lane * EPL < D;
    for (int s = 0; s < S; s++) {
        const size_t prow = base + (size_t)s * rows + row;
        const float2 ml = p.part_ml[prow];
        const float sc = exp2f(ml.x - Ms);
        ls = fmaf(sc, ml.y, ls);
        if (v_lane) {
            const float *po = p.part_o + prow * D + lane * EPL;
#pragma unroll
            for (int x = 0; x < EPL; x++) acc[x] = fmaf(sc, po[x], acc[x]);
        }
    }
    if (v_lane) {
        const int i = row / p.hq, h = row - (row / p.hq) * p.hq;
        __nv_bfloat16 *dst = p.out + ((size_t)(b + i) * p.hq + h) * D + lane * EPL;
#pragma unroll
        for (int x = 0; x < EPL; x++) dst[x] = __float2bfloat16(ls > 0.f ? acc[x] / ls : 0.f);
    }
}

cudaError_t launch_attn_combine(const AttnParams &p, const WorkList &wl, int head_dim,
                                int max_rows_per_req, cudaStream_t stream)
{
    if (wl.n <= 0) return cudaSuccess;
    dim3 grid(wl.n, (max_rows_per_req + 7) / 8);
    launch_begin(stream, kAttnCombine);
    cudaError_t e;
    switch (head_dim) {
    case 48: e = launch_maybe_pdl(attn_combine_kernel<48>, grid, dim3(256), 0, stream, p, wl); break;
    case 64: e = launch_maybe_pdl(attn_combine_kernel<64>, grid, dim3(256), 0, stream, p, wl); break;
    case 128: e = launch_maybe_pdl(attn_combine_kernel<128>, grid, dim3(256), 0, stream, p, wl); break;
    default: launch_end(stream); return cudaErrorInvalidValue;
    }
    launch_end(stream);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace pkv

// The split-KV reduction as a kernel of its own: merges the fp32 partials
// of split requests when they are not merged inside the attention kernels
// (a workspace without room for the split counters, warp-MMA prefill tiles
// split over keys).
#include "common.cuh"
#include "sm100.cuh"

namespace pkv {

// Split-KV combine pass.
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
    constexpr int EPL = D >= 128 ? 4 : 2;                 // output elements per lane
    const int li = blockIdx.x;
    const int b = wl.qb[li], t = wl.qt[li], L = wl.len[li];      // the planned length fixes the split count
    // decode-class requests split their (windowed) key range; every tile of a
    // split prefill request has ceil(L / split) splits
    const int S = wl.mode == kModeDecode ? decode_splits(t, L, p.window, wl.split_tokens)
                                         : (L + wl.split_tokens - 1) / wl.split_tokens;
    const int rows = t * p.hq;
    const int lane = threadIdx.x & 31;
    const int row = blockIdx.y * (blockDim.x / 32) + (threadIdx.x >> 5);
    pdl_wait();                                                   // the split partials are written
    if (row >= rows) return;
    if (run_len(p, wl, li) == 0) return;                          // a padding row at run time: zeros written
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

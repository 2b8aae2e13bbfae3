// indexer_simt.cuh -- lightning-indexer scores on the CUDA cores (fp32 FMA).
//
// DeepSeek-V4 hybrid attention, CSA step two (gxgjx.lffhtl.com/lxrt/355279.html, section
// 混肃穆力机制: a light indexer scores each query against every compressed block); [P4]
// section 3.1: 64 indexer heads of dim 128.  Score, as in the DeepSeek-V3.2 indexer:
//   s_j = sum_h w_h * ReLU(q_h . k_j)  for j < n_vis = floor((pos+1)/m), -inf beyond.
#pragma once

#include "common.cuh"

namespace lca {

constexpr int kIdxSimtRows = 128;

struct IndexerArgs {
    int HI, DI, ratio, n_q;
    const __nv_bfloat16 *q;      // [B][n_q][HI][DI]
    const float *w;              // [B][n_q][HI]
    const __nv_bfloat16 *k; int64_t k_bs; int64_t cache_rows;
    const int32_t *q_pos;        // [B][n_q]
    float *scores; int64_t s_stride;
};

// grid (ceil(cache_rows/128), n_q, B), block 128: thread t scores entry tile*128 + t.
__global__ void __launch_bounds__(kIdxSimtRows) indexer_simt_kernel(IndexerArgs a) {
    extern __shared__ __align__(16) float ism[];
    float *qs = ism;                          // [HI][DI]
    float *ws = qs + a.HI * a.DI;             // [HI]
    float *ks = ws + a.HI;                    // [DI][128] transposed tile
    const int b = blockIdx.z, qi = blockIdx.y;
    const int64_t row = (int64_t)b * a.n_q + qi;
    const int64_t pos = a.q_pos[row];
    int64_t n_vis = pos < 0 ? 0 : (pos + 1) / a.ratio;
    if (n_vis > a.cache_rows) {
        if (threadIdx.x == 0 && blockIdx.x == 0) raise_error(LCA_DEVERR_VISIBLE_RANGE);
        n_vis = a.cache_rows;
    }
    const int64_t j0 = (int64_t)blockIdx.x * kIdxSimtRows;
    const int64_t j = j0 + threadIdx.x;
    float *srow = a.scores + row * a.s_stride;
    if (j0 >= n_vis) {
        if (j < a.cache_rows) srow[j] = -INFINITY;
        return;
    }
    const __nv_bfloat16 *qp = a.q + row * a.HI * a.DI;
    for (int i = threadIdx.x; i < a.HI * a.DI; i += blockDim.x) qs[i] = __bfloat162float(qp[i]);
    for (int i = threadIdx.x; i < a.HI; i += blockDim.x) ws[i] = a.w[row * a.HI + i];
    const __nv_bfloat16 *kp = a.k + (int64_t)b * a.k_bs;
    for (int i = threadIdx.x; i < kIdxSimtRows * a.DI; i += blockDim.x) {
        const int r = i / a.DI, d = i % a.DI;
        const int64_t jj = j0 + r;
        ks[d * kIdxSimtRows + r] = jj < n_vis ? __bfloat162float(kp[jj * a.DI + d]) : 0.f;
    }
    __syncthreads();
    if (j >= a.cache_rows) return;
    if (j >= n_vis) {
        srow[j] = -INFINITY;
        return;
    }
    float s = 0.f;
    for (int h = 0; h < a.HI; ++h) {
        float dot = 0.f;
        for (int d = 0; d < a.DI; ++d) dot = fmaf(qs[h * a.DI + d], ks[d * kIdxSimtRows + threadIdx.x], dot);
        s = fmaf(ws[h], fmaxf(dot, 0.f), s);
    }
    srow[j] = s;
}

}  // namespace lca

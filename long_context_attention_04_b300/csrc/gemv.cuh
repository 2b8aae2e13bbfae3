// gemv.cuh -- small-batch products C[M][N] = A[M][K] . B[N][K]^T for M <= 16 (decode).
//
// Used by the grouped output projection (DeepSeek-V4 CSA step four, gxgjx.lffhtl.com/lxrt/
// 355279.html section 混肃穆力机制: heads split into g groups, each projected to d_g, then
// merged to d).  At decode batch sizes the product streams the weight matrix B once from
// HBM and does M multiply-adds per weight, far below the tensor-core ridge, so it stays on
// the CUDA cores: each warp owns 4 weight rows, reads them with 16-byte loads (a warp reads
// 512 contiguous bytes of a row per step, several steps loaded before the first multiply)
// and keeps M x 4 fp32 accumulators.
#pragma once

#include "common.cuh"

namespace lca {

constexpr int kGemvThreads = 256;
constexpr int kGemvRowsPerWarp = 4;

// 256-element steps loaded ahead per iteration: fewer for larger M (registers)
template <int MT>
__host__ __device__ constexpr int gemv_unroll() { return MT <= 4 ? 4 : MT <= 8 ? 2 : 1; }

struct GemvArgs {
    int M, N, K;
    const __nv_bfloat16 *A; int64_t lda; int64_t a_batch_off;
    const __nv_bfloat16 *B; int64_t ldb; int64_t b_batch_off;
    __nv_bfloat16 *C; int64_t ldc; int64_t c_batch_off;
};

// grid (ceil(N / (8 warps * 4 rows)), batches), block 256.
template <int MT>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(GemvArgs a) {
    pdl_trigger();
    pdl_wait();
    constexpr int U = gemv_unroll<MT>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n0 = ((int64_t)blockIdx.x * (kGemvThreads / 32) + warp) * kGemvRowsPerWarp;
    if (n0 >= a.N) return;
    const __nv_bfloat16 *A = a.A + blockIdx.y * a.a_batch_off;
    const __nv_bfloat16 *B = a.B + blockIdx.y * a.b_batch_off;
    __nv_bfloat16 *C = a.C + blockIdx.y * a.c_batch_off;
    float acc[MT][kGemvRowsPerWarp];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < kGemvRowsPerWarp; ++r) acc[m][r] = 0.f;
    const int nrows = (a.N - n0) < kGemvRowsPerWarp ? (int)(a.N - n0) : kGemvRowsPerWarp;
    for (int k0 = lane * 8; k0 < a.K; k0 += 32 * 8 * U) {
        uint4 wv[U][kGemvRowsPerWarp], av[U][MT];
#pragma unroll
        for (int s = 0; s < U; ++s) {
            const int k = k0 + s * 32 * 8;
#pragma unroll
            for (int r = 0; r < kGemvRowsPerWarp; ++r)
                wv[s][r] = (k < a.K && r < nrows) ? __ldg(reinterpret_cast<const uint4 *>(B + (n0 + r) * a.ldb + k))
                                                 : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int m = 0; m < MT; ++m)
                av[s][m] = (k < a.K && m < a.M) ? __ldg(reinterpret_cast<const uint4 *>(A + m * a.lda + k))
                                                : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int s = 0; s < U; ++s) {
#pragma unroll
            for (int r = 0; r < kGemvRowsPerWarp; ++r) {
                float bw[8];
                unpack8(wv[s][r], bw);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float x[8];
                    unpack8(av[s][m], x);
#pragma unroll
                    for (int u = 0; u < 8; ++u) acc[m][r] = fmaf(x[u], bw[u], acc[m][r]);
                }
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < kGemvRowsPerWarp; ++r) acc[m][r] = warp_sum(acc[m][r]);
    if (lane == 0) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < kGemvRowsPerWarp; ++r)
                if (m < a.M && r < nrows) C[m * a.ldc + n0 + r] = __float2bfloat16_rn(acc[m][r]);
    }
}

}  // namespace lca

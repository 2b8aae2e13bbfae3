// gemv.cuh -- small-batch products C[M][N] = A[M][K] . B[N][K]^T for M <= 16 (decode).
//
// Used by the grouped output projection (DeepSeek-V4 CSA step four, gxgjx.lffhtl.com/lxrt/
// 355279.html section 混肃穆力机制: heads split into g groups, each projected to d_g, then
// merged to d).  At decode batch sizes the product streams the weight matrix B once from
// HBM and does M multiply-adds per weight, far below the tensor-core ridge, so it stays on
// the CUDA cores: each warp owns 4 weight rows, reads them with 16-byte loads (a warp reads
// 512 contiguous bytes of a row per step) and keeps M x 4 fp32 accumulators.
#pragma once

#include "common.cuh"

namespace lca {

constexpr int kGemvThreads = 256;
constexpr int kGemvRowsPerWarp = 4;

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
    for (int k = lane * 8; k < a.K; k += 32 * 8) {
        float bw[kGemvRowsPerWarp][8];
#pragma unroll
        for (int r = 0; r < kGemvRowsPerWarp; ++r) {
            if (r < nrows) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(B + (n0 + r) * a.ldb + k));
                unpack8(v, bw[r]);
            } else {
#pragma unroll
                for (int u = 0; u < 8; ++u) bw[r][u] = 0.f;
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
            if (m < a.M) {
                float av[8];
                unpack8(__ldg(reinterpret_cast<const uint4 *>(A + m * a.lda + k)), av);
#pragma unroll
                for (int r = 0; r < kGemvRowsPerWarp; ++r)
#pragma unroll
                    for (int u = 0; u < 8; ++u) acc[m][r] = fmaf(av[u], bw[r][u], acc[m][r]);
            }
        }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < kGemvRowsPerWarp; ++r) acc[m][r] = warp_sum(acc[m][r]);
    if (lane == 0) {
        for (int m = 0; m < a.M; ++m)
            for (int r = 0; r < nrows; ++r) C[m * a.ldc + n0 + r] = __float2bfloat16_rn(acc[m][r]);
    }
}

}  // namespace lca

// mhc.cuh -- manifold-constrained hyper-connections (DeepSeek-V4, gxgjx.lffhtl.com/lxrt/
// 355279.html section "mHC，给残差集结加层连续"; zhinnengdao.top section 3.2 "mHC"): the
// residual stream is n parallel streams x[i] of width d; per token and layer, n pre-weights a
// and n post-weights c (sigmoids) and an n x n mixing matrix B are generated from the input,
// B projected onto the doubly stochastic matrices by Sinkhorn-Knopp (row and column
// normalisations in turn, `iters` times; 20 on the page).  The layer reads h = sum_i a_i x[i];
// after it, x'[i] = sum_j B[i][j] x[j] + c_i y with y the layer's output.
//
// The generated values z = flatten(x) . Phi^T (2n + n^2 per token) come from the tensor-core
// product (gemm_tc.cuh), whose epilogue thread for a token row holds all of that token's values
// in registers: it adds the bias and computes the sigmoids and the Sinkhorn-Knopp iteration
// there (mhc_coeffs_thread), so the iteration's latency is spread over 128 tokens per CTA and
// nothing is written but the coefficients.  The stream mixings (mhc_pre_mix_kernel for h,
// mhc_post_kernel for the new streams) are then plain streaming kernels: one thread per
// 8-element chunk of a token, 16-byte loads and stores, fp32 arithmetic.
#pragma once

#include "common.cuh"

namespace lca {

constexpr int kMhcThreads = 256;

// Where the product's epilogue puts the coefficients (one token per row of the product).
struct MhcCoeffArgs {
    const float *bias;        // [2n + n^2]
    float *a, *c, *B;         // [T][n], [T][n], [T][n][n]
    int iters;
};

// Token t's coefficients from its generated values z[0 .. 2n + n^2) (bias not yet added).
template <int N>
__device__ __forceinline__ void mhc_coeffs_thread(const uint32_t *zv, int64_t t, const MhcCoeffArgs &m) {
    constexpr int K = 2 * N + N * N;
    float z[K];
#pragma unroll
    for (int k = 0; k < K; ++k) z[k] = __uint_as_float(zv[k]) + __ldg(m.bias + k);
#pragma unroll
    for (int i = 0; i < N; ++i) {
        m.a[t * N + i] = 1.f / (1.f + expf(-z[i]));
        m.c[t * N + i] = 1.f / (1.f + expf(-z[N + i]));
    }
    // exp of each row less its maximum: the first row normalisation divides the row's common
    // factor out again, so the iteration gives the result of exp(z) without its overflow
    float b[N * N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        float mx = z[2 * N + i * N];
#pragma unroll
        for (int j = 1; j < N; ++j) mx = fmaxf(mx, z[2 * N + i * N + j]);
#pragma unroll
        for (int j = 0; j < N; ++j) b[i * N + j] = expf(z[2 * N + i * N + j] - mx);
    }
    for (int it = 0; it < m.iters; ++it) {
#pragma unroll
        for (int i = 0; i < N; ++i) {          // rows
            float s = 0.f;
#pragma unroll
            for (int j = 0; j < N; ++j) s += b[i * N + j];
            const float r = 1.f / s;
#pragma unroll
            for (int j = 0; j < N; ++j) b[i * N + j] *= r;
        }
#pragma unroll
        for (int j = 0; j < N; ++j) {          // columns
            float s = 0.f;
#pragma unroll
            for (int i = 0; i < N; ++i) s += b[i * N + j];
            const float r = 1.f / s;
#pragma unroll
            for (int i = 0; i < N; ++i) b[i * N + j] *= r;
        }
    }
#pragma unroll
    for (int e = 0; e < N * N; ++e) m.B[t * N * N + e] = b[e];
}

struct MhcMixArgs {
    int d;
    const __nv_bfloat16 *x;   // [T][n][d]
    const float *a, *c, *B;   // coefficients
    __nv_bfloat16 *h;         // [T][d]
    const __nv_bfloat16 *y;   // [T][d]
    __nv_bfloat16 *x_out;     // [T][n][d]
};

// grid (ceil(d / 8 / 256), T): h[t][e..e+8) = sum_i a[t][i] x[t][i][e..e+8).
template <int N>
__global__ void __launch_bounds__(kMhcThreads) mhc_pre_mix_kernel(MhcMixArgs m) {
    pdl_trigger();
    pdl_wait();
    const int64_t t = blockIdx.y;
    const int e = 8 * (blockIdx.x * kMhcThreads + threadIdx.x);
    if (e >= m.d) return;
    const __nv_bfloat16 *xt = m.x + t * N * (int64_t)m.d + e;
    uint4 xv[N];
#pragma unroll
    for (int i = 0; i < N; ++i) xv[i] = __ldg(reinterpret_cast<const uint4 *>(xt + (int64_t)i * m.d));
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float ai = __ldg(m.a + t * N + i);
        float f[8];
        unpack8(xv[i], f);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = fmaf(ai, f[k], acc[k]);
    }
    *reinterpret_cast<uint4 *>(m.h + t * (int64_t)m.d + e) = pack8(acc);
}

// grid (ceil(d / 8 / 256), T): x'[t][i][e..e+8) = sum_j B[t][i][j] x[t][j][e..e+8) + c[t][i] y[t][e..e+8).
template <int N>
__global__ void __launch_bounds__(kMhcThreads) mhc_post_kernel(MhcMixArgs m) {
    pdl_trigger();
    pdl_wait();
    const int64_t t = blockIdx.y;
    const int e = 8 * (blockIdx.x * kMhcThreads + threadIdx.x);
    if (e >= m.d) return;
    const __nv_bfloat16 *xt = m.x + t * N * (int64_t)m.d + e;
    float xs[N][8], yv[8];
#pragma unroll
    for (int j = 0; j < N; ++j) unpack8(__ldg(reinterpret_cast<const uint4 *>(xt + (int64_t)j * m.d)), xs[j]);
    unpack8(__ldg(reinterpret_cast<const uint4 *>(m.y + t * (int64_t)m.d + e)), yv);
    __nv_bfloat16 *ot = m.x_out + t * N * (int64_t)m.d + e;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float ci = __ldg(m.c + t * N + i);
        float bi[N];
#pragma unroll
        for (int j = 0; j < N; ++j) bi[j] = __ldg(m.B + (t * N + i) * N + j);
        float o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float s = ci * yv[k];
#pragma unroll
            for (int j = 0; j < N; ++j) s = fmaf(bi[j], xs[j][k], s);
            o[k] = s;
        }
        *reinterpret_cast<uint4 *>(ot + (int64_t)i * m.d) = pack8(o);
    }
}

}  // namespace lca

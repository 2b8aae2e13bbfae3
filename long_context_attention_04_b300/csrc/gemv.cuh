// gemv.cuh -- small-batch products C[M][N] = A[M][K] . B[N][K]^T for M <= 16 (decode).
//
// Used by the grouped output projection (DeepSeek-V4 CSA step four, gxgjx.lffhtl.com/lxrt/
// 355279.html section 混肃穆力机制: heads split into g groups, each projected to d_g, then
// merged to d).  At decode batch sizes the product streams the weight matrix B once from
// HBM and does M multiply-adds per weight, far below the tensor-core ridge, so it stays on
// the CUDA cores: each warp owns 4 weight rows, reads them with 16-byte loads (a warp reads
// 512 contiguous bytes of a row per step, several steps loaded before the first multiply)
// and keeps M x 4 fp32 accumulators.
//
// gemv_stream_kernel is the bandwidth path for weight matrices stored as one contiguous
// array (the grouped projections' Wg and Wm): one CTA per SM streams its share of the weight
// rows through a shared-memory ring with 1D bulk copies (32-64 KB each, 128-192 KB in
// flight), which holds HBM near its copy rate where per-thread 16-byte loads stall at a
// third of it.  The activations stay in registers: consumer warp w owns a fixed slice of
// the K dimension for every row, so it loads its slice of A once and reuses it for all the
// rows; per 4-row chunk each warp reduces its 4 x M partial sums across lanes (a butterfly
// that hands each lane one of the sums), and the 8 warps' partials are added in a fixed order
// (the result does not depend on timing).
#pragma once

#include "common.cuh"
#include "ptx.cuh"

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

// ------------------------------------------------------------------ streaming path ---

constexpr int kGsRows = 4;                                // weight rows per ring stage
constexpr int kGsRingBytes = 196608;                      // ring capacity (stages of 8 K bytes)
constexpr int kGsMaxStages = 8;

struct GemvStreamArgs {
    int M, N, K;
    int64_t groups;            // 4-row groups over all batches: batches * N / 4
    const __nv_bfloat16 *A; int64_t lda; int64_t a_batch_off;
    const __nv_bfloat16 *B;    // [batches][N][K], contiguous
    __nv_bfloat16 *C; int64_t ldc; int64_t c_batch_off;
    int b_early;               // B may be read before the previous kernel in the stream completes
};

__host__ __device__ constexpr int gemv_stream_stages(int K) {
    return kGsRingBytes / (kGsRows * K * 2) < kGsMaxStages ? kGsRingBytes / (kGsRows * K * 2) : kGsMaxStages;
}
// dynamic shared memory: 1 KB alignment pad + ring + mbarriers + partial-sum slots
__host__ __device__ constexpr int gemv_stream_smem(int K, int MT, int NW) {
    return 1024 + gemv_stream_stages(K) * kGsRows * K * 2 + kGsMaxStages * 8 + 2 * NW * kGsRows * MT * 4;
}

// Sum V = 2^P values across the warp: afterwards every lane holds the warp total of value
// index (lane >> (5 - P)), in v[0].  P halving steps (each lane keeps the half its lane bit
// selects and adds its partner's copy of that half), then 5 - P steps over the lanes that
// ended with the same index.
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[V]) {
    constexpr int P = V == 32 ? 5 : V == 16 ? 4 : V == 8 ? 3 : V == 4 ? 2 : V == 2 ? 1 : 0;
    static_assert((1 << P) == V, "V must be a power of two <= 32");
#pragma unroll
    for (int step = 0; step < P; ++step) {
        const int n = V >> step, o = 16 >> step;
        const bool upper = (threadIdx.x & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
#pragma unroll
    for (int o = 16 >> P; o >= 1; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
    return v[0];
}

// grid: one CTA per SM (at most `groups`), block 32 NW, dynamic smem gemv_stream_smem.
// CTA i owns the 4-row groups [i G / grid, (i + 1) G / grid): contiguous weight bytes, copied
// a group (one ring stage) at a time by thread 0.  A stage is refilled right after the
// block-wide barrier that ends its group, when every warp has finished reading it.
template <int MT, int KS, int NW>
__global__ void __launch_bounds__(32 * NW, 1) gemv_stream_kernel(GemvStreamArgs a) {
    using namespace ptx;
    constexpr int K = KS * 256 * NW;                          // row length (elements)
    constexpr int STAGE = kGsRows * K * 2;
    constexpr int STAGES = gemv_stream_stages(K);
    constexpr int V = kGsRows * MT;                           // partial sums per group and warp
    constexpr int SH = V == 32 ? 0 : V == 16 ? 1 : V == 8 ? 2 : V == 4 ? 3 : 4;   // 5 - log2(V)
    extern __shared__ uint8_t gs_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(gs_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(ring + STAGES * STAGE);
    float *slots = reinterpret_cast<float *>(full + kGsMaxStages);   // [2][warps][V]
    pdl_trigger();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t g0 = (int64_t)blockIdx.x * a.groups / gridDim.x;
    const int64_t g1 = (int64_t)(blockIdx.x + 1) * a.groups / gridDim.x;
    const int nch = (int)(g1 - g0);
    int issued = 0;
    auto issue = [&](int j) {
        const int s = j % STAGES;
        mbar_arrive_expect_tx(&full[s], STAGE);
        bulk_load(smem_u32(ring + s * STAGE), a.B + (g0 + j) * (int64_t)(kGsRows * K), STAGE, &full[s]);
    };
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
        if (a.b_early)
            for (; issued < STAGES && issued < nch; ++issued) issue(issued);
    }
    __syncthreads();
    pdl_wait();
    if (threadIdx.x == 0)
        for (; issued < STAGES && issued < nch; ++issued) issue(issued);

    // warp w owns the K slice [w KS 256, (w + 1) KS 256) of every row
    const int kw = warp * KS * 256 + lane * 8;
    float af[MT][KS][8];
    int64_t cur_batch = -1;
    bool ok = true;
    int failed_at = -1;
    for (int j = 0; j < nch; ++j) {
        const int64_t r0 = (g0 + j) * kGsRows;
        const int64_t batch = r0 / a.N;
        const int64_t n0 = r0 - batch * a.N;
        if (batch != cur_batch) {
            cur_batch = batch;
            const __nv_bfloat16 *A = a.A + batch * a.a_batch_off;
#pragma unroll
            for (int m = 0; m < MT; ++m)
#pragma unroll
                for (int s = 0; s < KS; ++s) {
                    const uint4 v = m < a.M ? __ldg(reinterpret_cast<const uint4 *>(A + m * a.lda + kw + s * 256))
                                            : make_uint4(0u, 0u, 0u, 0u);
                    unpack8(v, af[m][s]);
                }
        }
        const int st = j % STAGES;
        if (ok && !mbar_wait(&full[st], (j / STAGES) & 1)) {
            ok = false;
            failed_at = j;
        }
        float acc[V];
#pragma unroll
        for (int i = 0; i < V; ++i) acc[i] = 0.f;
        if (ok) {
            const uint8_t *stage = ring + st * STAGE;
#pragma unroll
            for (int s = 0; s < KS; ++s)
#pragma unroll
                for (int r = 0; r < kGsRows; ++r) {
                    float w[8];
                    unpack8(*reinterpret_cast<const uint4 *>(stage + ((int64_t)r * K + kw + s * 256) * 2), w);
#pragma unroll
                    for (int m = 0; m < MT; ++m)
#pragma unroll
                        for (int u = 0; u < 8; ++u) acc[r * MT + m] = fmaf(af[m][s][u], w[u], acc[r * MT + m]);
                }
        }
        const float tot = warp_reduce_scatter<V>(acc);
        float *slot = slots + (j & 1) * NW * V;
        if ((lane & ((1 << SH) - 1)) == 0) slot[warp * V + (lane >> SH)] = tot;
        __syncthreads();   // every warp is done with stage st and has written its partials
        if (threadIdx.x == 0 && ok && issued < nch) issue(issued++);
        if (warp == j % NW && lane < V) {
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < NW; ++w) sum += slot[w * V + lane];
            const int r = lane / MT, m = lane % MT;
            if (ok && m < a.M) a.C[batch * a.c_batch_off + m * a.ldc + n0 + r] = __float2bfloat16_rn(sum);
        }
    }
    // after a timed-out wait the copies still in flight must land before the CTA exits
    if (threadIdx.x == 0 && failed_at >= 0)
        for (int j = failed_at; j < issued; ++j)
            if (!mbar_wait(&full[j % STAGES], (j / STAGES) & 1)) break;
}

}  // namespace lca

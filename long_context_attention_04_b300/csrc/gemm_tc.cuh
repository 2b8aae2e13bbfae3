// gemm_tc.cuh -- C[M][N] = A[M][K] . B[N][K]^T on the tcgen05 tensor cores, for products with
// many rows: the input projections of a prefill chunk (DeepSeek-V4 hybrid attention,
// gxgjx.lffhtl.com/lxrt/355279.html section 混肃穆力机制: the layers' queries, indexer
// queries and KV tokens are linear maps of the hidden state) and the dynamic parameters of
// the manifold-constrained hyper-connections (same page, section mHC: the mixing
// coefficients are generated from the layer input by a learned linear map).  Small-batch
// products (M <= 16, decode) stay on gemv.cuh: there the weights are read once and the
// tensor cores would idle.
//
// One CTA per 128 x BN output tile: a TMA warp streams 128 x 64 tiles of A and BN x 64 tiles
// of B (both K-major, 128-byte swizzled) through a multi-stage shared-memory ring, one thread
// issues tcgen05.mma (M = 128, N = BN, K = 16, bf16 in, fp32 accumulation in TMEM), and four
// epilogue warps (one per TMEM lane quarter) read the accumulator and store fp32 or bf16
// rows.  Out-of-range rows and K columns of a tile are read as zeros by the TMA unit and
// out-of-range outputs are not stored, so M, N and K need no padding (K a multiple of 8:
// 16-byte rows).  Every wait is bounded (LCA_DEVERR_TIMEOUT).  With MHC_N > 0 the product is
// the hyper-connections' generated values (N = 2n + n^2 <= 32 columns) and the epilogue turns
// each token row into its coefficients (mhc_coeffs_thread) instead of storing it.
#pragma once

#include "common.cuh"
#include "mhc.cuh"
#include "ptx.cuh"

namespace lca {

constexpr int kGtBM = 128, kGtBK = 64;
constexpr int kGtThreads = 192;          // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue

template <int BN>
struct GemmTcConfig {
    static constexpr int A_BYTES = kGtBM * kGtBK * 2;                  // 16 KB
    static constexpr int B_BYTES = BN * kGtBK * 2;
    static constexpr int STAGES = BN >= 256 ? 4 : BN >= 128 ? 6 : 8;
    static constexpr int MISC = 256;
    static constexpr int SMEM_BYTES = MISC + 1024 + STAGES * (A_BYTES + B_BYTES);
    static constexpr int TMEM_COLS = BN < 32 ? 32 : BN;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

struct GemmTcArgs {
    int M, N, K;
    void *C;                // fp32 or bf16 rows of ldc elements
    int64_t ldc;
    MhcCoeffArgs mhc;       // MHC_N > 0 only
};

template <int BN, bool F32_OUT, int MHC_N = 0>
__global__ void __launch_bounds__(kGtThreads) gemm_tc_kernel(const __grid_constant__ CUtensorMap a_map,
                                                           const __grid_constant__ CUtensorMap b_map, GemmTcArgs g) {
    using Cfg = GemmTcConfig<BN>;
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_raw);
    uint64_t *empty = full + Cfg::STAGES;
    uint64_t *acc_full = empty + Cfg::STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_full + 1);
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw + Cfg::MISC) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *a_ring = base;
    uint8_t *b_ring = base + Cfg::STAGES * Cfg::A_BYTES;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(acc_full, 1);
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();
    const int n0 = blockIdx.x * BN, m0 = blockIdx.y * kGtBM;
    const int ksteps = (g.K + kGtBK - 1) / kGtBK;
    bool ok = true;
    if (warp == 0) {
        if (lane == 0) {
            ptx::tma_prefetch(&a_map);
            ptx::tma_prefetch(&b_map);
            int issued = 0;
            for (int k = 0; k < ksteps; ++k) {
                const int s = k % Cfg::STAGES;
                if (k >= Cfg::STAGES && !ptx::mbar_wait(&empty[s], ((k / Cfg::STAGES) - 1) & 1)) {
                    ok = false;
                    break;
                }
                ptx::mbar_arrive_expect_tx(&full[s], Cfg::A_BYTES + Cfg::B_BYTES);
                ptx::tma_load_2d(ptx::smem_u32(a_ring + s * Cfg::A_BYTES), &a_map, k * kGtBK, m0, &full[s]);
                ptx::tma_load_2d(ptx::smem_u32(b_ring + s * Cfg::B_BYTES), &b_map, k * kGtBK, n0, &full[s]);
                issued = k + 1;
            }
            // copies still landing when the CTA exits would write freed shared memory: wait for
            // the last one issued into each stage (these phases have normally been seen already)
            for (int k = issued - 1; k >= 0 && k >= issued - Cfg::STAGES; --k)
                ptx::mbar_wait(&full[k % Cfg::STAGES], (k / Cfg::STAGES) & 1);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = ptx::idesc_bf16(kGtBM, BN, false, false);
            const uint64_t a_d = ptx::smem_desc(ptx::smem_u32(a_ring), 16, 1024, ptx::kSwizzle128);
            const uint64_t b_d = ptx::smem_desc(ptx::smem_u32(b_ring), 16, 1024, ptx::kSwizzle128);
            for (int k = 0; k < ksteps; ++k) {
                const int s = k % Cfg::STAGES;
                if (!ptx::mbar_wait(&full[s], (k / Cfg::STAGES) & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kGtBK / 16; ++kk)
                    ptx::mma_bf16(tmem, a_d + (uint64_t)(s * (Cfg::A_BYTES >> 4) + kk * 2),
                                  b_d + (uint64_t)(s * (Cfg::B_BYTES >> 4) + kk * 2), idesc, (k > 0 || kk > 0) ? 1u : 0u);
                ptx::mma_commit(&empty[s]);
            }
            ptx::mma_commit(acc_full);   // also the teardown point: every issued MMA completes first
            ptx::mbar_wait(acc_full, 0);
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 = tile rows
        const int q = warp & 3;
        if (ptx::mbar_wait(acc_full, 0)) {
            ptx::tc_fence_after();
            const int row = m0 + 32 * q + lane;
            if constexpr (MHC_N > 0) {
                // one token per row: its 2n + n^2 generated values are columns 0 .. 31 of the tile
                uint32_t v[32];
                ptx::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16), v);
                ptx::tmem_ld_wait();
                if (row < g.M) mhc_coeffs_thread<MHC_N>(v, row, g.mhc);
            } else
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                uint32_t v[32];
                ptx::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + c0, v);
                ptx::tmem_ld_wait();
                if (row < g.M) {
                    const int ncol = g.N - (n0 + c0);
                    if (F32_OUT) {
                        float *dst = static_cast<float *>(g.C) + (int64_t)row * g.ldc + n0 + c0;
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (i < ncol) dst[i] = __uint_as_float(v[i]);
                    } else {
                        __nv_bfloat16 *dst = static_cast<__nv_bfloat16 *>(g.C) + (int64_t)row * g.ldc + n0 + c0;
                        if ((reinterpret_cast<uintptr_t>(dst) & 3) == 0) {   // pairs of columns per store
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                if (i + 1 < ncol)
                                    *reinterpret_cast<uint32_t *>(dst + i) =
                                        pack_bf16x2(__uint_as_float(v[i]), __uint_as_float(v[i + 1]));
                                else if (i < ncol)
                                    dst[i] = __float2bfloat16_rn(__uint_as_float(v[i]));
                            }
                        } else {                                              // an odd row start (odd ldc)
#pragma unroll
                            for (int i = 0; i < 32; ++i)
                                if (i < ncol) dst[i] = __float2bfloat16_rn(__uint_as_float(v[i]));
                        }
                    }
                }
            }
            ptx::tc_fence_before();
        }
    }
    (void)ok;
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

}  // namespace lca

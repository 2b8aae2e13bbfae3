// quant.cuh -- per-row e4m3 quantisation of bf16 rows, for FP8 compressed caches and FP8
// indexer queries (a variant of the path: the pages name FP8 storage only in passing --
// ynrysl.com, the paragraph on HCA -- and give no format; the reading taken is one fp32 scale
// per row, the row's largest magnitude mapped to 448, the largest finite e4m3 value):
//     scale = amax / 448,   code_i = e4m3(x_i / scale)   (IEEE fp32 divisions, round to
//     nearest even, saturating), read back as scale * e4m3_value(code_i).
// An all-zero row gets scale 0 and zero codes.
//
// Bandwidth-trivial: one warp per row, 16-byte loads, the row kept in registers between the
// amax reduction and the conversion, 8-byte code stores.
#pragma once

#include "common.cuh"

namespace lca {

constexpr int kQuantWarps = 8;           // rows per CTA
constexpr int kQuantMaxChunks = 4;       // 16-byte chunks per lane: width <= 32 * 4 * 8 = 1024

struct QuantArgs {
    const __nv_bfloat16 *x;
    int64_t rows;
    int width;                           // multiple of 8, <= 1024
    uint8_t *q;                          // [rows][width]
    float *scale;                        // [rows]
};

// grid ceil(rows / kQuantWarps), block 32 * kQuantWarps.
__global__ void __launch_bounds__(32 * kQuantWarps) quantize_rows_kernel(QuantArgs a) {
    pdl_trigger();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = (int64_t)blockIdx.x * kQuantWarps + warp;
    if (r >= a.rows) return;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.x + r * a.width);
    const int chunks = a.width / 8;
    float f[kQuantMaxChunks][8];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kQuantMaxChunks; ++i) {
        const int c = lane + 32 * i;
        if (c < chunks) {
            unpack8(__ldg(src + c), f[i]);
#pragma unroll
            for (int u = 0; u < 8; ++u) amax = fmaxf(amax, fabsf(f[i][u]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(amax, 448.f);
    if (lane == 0) a.scale[r] = s;
    uint2 *dst = reinterpret_cast<uint2 *>(a.q + r * a.width);
#pragma unroll
    for (int i = 0; i < kQuantMaxChunks; ++i) {
        const int c = lane + 32 * i;
        if (c < chunks) dst[c] = amax > 0.f ? e4m3x8(f[i], s) : make_uint2(0u, 0u);
    }
}

}  // namespace lca

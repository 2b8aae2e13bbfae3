// q_prep.cuh -- the query side of core attention, computed once per query for all its
// split-K CTAs: RMSNorm over c with gamma_q ("Q/KV normalization"), RoPE at the query
// position on the trailing R dims ("Partial RoPE"), then the split q = hi + lo into two fp16
// parts (DeepSeek-V4 hybrid attention, gxgjx.lffhtl.com/lxrt/355279.html, section 混肃穆力机制).
//
// Output: per query, an image of [c/128 chunks][2 boxes of 64 c][128 rows][128 bytes],
// 128-byte swizzled (16-byte chunk index XOR row % 8): the shared-memory layout of a K-major
// tcgen05.mma operand with 128 rows.  Row 32 g + i holds the hi part of head 16 g + i and row
// 32 g + 16 + i its lo part (g < 4, i < 16), so that the two parts of a head land in the same
// 32-lane quarter of tensor memory, 16 lanes apart, when the attention kernel moves the image
// there as the A operand of its logit product.  Heads past H are zero rows.  hi + lo carries the
// normalised query to about 22 bits (fp16 keeps 11 each); an element beyond fp16's range is
// reported (LCA_DEVERR_FP16_RANGE).
#pragma once

#include "attend_common.cuh"

namespace lca {

constexpr int kQPrepHeads = 8;              // heads (warps) per CTA
constexpr int kQImgHeads = 64;              // padded heads of an image

constexpr int kQChunkBytes = 2 * 128 * 128;   // one c chunk of the image: 2 boxes x 128 rows x 128 B

template <int C>
__device__ __forceinline__ uint8_t *q_img(const AttendArgs &a, int64_t unit) {
    return a.q_img + unit * (int64_t)((C / 128) * kQChunkBytes);
}

__host__ __device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
    return row * 128u + (((chunk ^ (row & 7u)) & 7u) << 4);
}

// Image row of head h's hi (part 0) or lo (part 1) half.
__host__ __device__ __forceinline__ uint32_t q_img_row(uint32_t h, uint32_t part) {
    return 32u * (h >> 4) + 16u * part + (h & 15u);
}

// grid (units, 64 / kQPrepHeads), block 32 * kQPrepHeads: warp w prepares head blockIdx.y*8 + w.
template <int C>
__global__ void __launch_bounds__(32 * kQPrepHeads) q_prep_kernel(AttendArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ float rcs[64], rsn[64];
    const int64_t unit = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y * kQPrepHeads + warp;
    constexpr int EPL = C / 32;
    QLane<C> ql;
    if (h < a.H) q_load_warp<C>(a, a.q + (unit * a.H + h) * C, ql);   // in flight during the RoPE table
    int64_t pos = a.q_pos[unit];
    if (pos < 0) pos = 0;
    rope_table_fill(a, pos, rcs, rsn);
    __syncthreads();
    float v[EPL];
    if (h < a.H) {
        q_hat_warp<C>(a, ql, rcs, rsn, v);
    } else {
#pragma unroll
        for (int u = 0; u < EPL; ++u) v[u] = 0.f;
    }
    // an element outside fp16's finite range would saturate in the image: reported, not hidden
    bool bad = false;
#pragma unroll
    for (int u = 0; u < EPL; ++u) bad |= !(fabsf(v[u]) <= 65504.f);
    if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(LCA_DEVERR_FP16_RANGE);
    float lo[EPL];
#pragma unroll
    for (int u = 0; u < EPL; ++u) {
        const float hi = __half2float(__float2half_rn(v[u]));
        lo[u] = v[u] - hi;
        v[u] = hi;
    }
    uint8_t *img = q_img<C>(a, unit);
    // element e of head h: chunk e/128, box (e%128)/64, rows h (hi) and 64 + h (lo)
    if constexpr (EPL >= 8) {
#pragma unroll
        for (int u = 0; u < EPL; u += 8) {
            const int e = lane * EPL + u;
            uint8_t *box = img + (e / 128) * kQChunkBytes + ((e % 128) / 64) * (128 * 128);
            *reinterpret_cast<uint4 *>(box + sw128(q_img_row(h, 0), (e % 64) / 8)) = pack8_f16(v + u);
            *reinterpret_cast<uint4 *>(box + sw128(q_img_row(h, 1), (e % 64) / 8)) = pack8_f16(lo + u);
        }
    } else {
        const int e = lane * EPL;   // 4 elements: half a 16-byte chunk
        uint8_t *box = img + (e / 128) * kQChunkBytes + ((e % 128) / 64) * (128 * 128) + (e % 8) * 2;
        *reinterpret_cast<uint2 *>(box + sw128(q_img_row(h, 0), (e % 64) / 8)) =
            make_uint2(pack_f16x2(v[0], v[1]), pack_f16x2(v[2], v[3]));
        *reinterpret_cast<uint2 *>(box + sw128(q_img_row(h, 1), (e % 64) / 8)) =
            make_uint2(pack_f16x2(lo[0], lo[1]), pack_f16x2(lo[2], lo[3]));
    }
}

}  // namespace lca

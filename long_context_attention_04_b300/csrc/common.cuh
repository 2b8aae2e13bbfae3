// common.cuh -- device helpers shared by the kernels of liblca (bf16 packing, the device
// error word, block reductions, RoPE angles).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lca.h"

namespace lca {

// One error word per device (the library is a single translation unit).  Kernels OR
// LCA_DEVERR_* bits into it; lca_device_error() reads and clears it.
__device__ unsigned int g_error_word;

__device__ __forceinline__ void raise_error(unsigned int bits) { atomicOr(&g_error_word, bits); }

// Bound of every mbarrier wait, in SM clock cycles (~1 s at 2 GHz by default), and a tile the
// attention kernel's producer leaves unloaded (-1: none).  Both are changed only through
// lca_test_hooks, which tests use to make a wait run out on purpose; kernels read them once
// per launch (the skip) or once per slow wait (the bound).
__device__ long long g_wait_limit_cycles = 2000000000LL;
__device__ int g_test_skip_tile = -1;

// Programmatic dependent launch.  Every kernel of the library is launched so that the next
// kernel in the stream may be scheduled while it runs (its CTAs then wait on the SMs instead
// of behind a launch).  Each kernel calls pdl_trigger() first, to let the next one launch,
// and pdl_wait() before its first access to global memory, on every path: pdl_wait returns
// once the previous kernel in the stream has completed and its writes are visible, and
// because every kernel waits before it can complete, completion stays ordered along the
// whole stream.  One documented exception: the grouped output projection starts reading its
// weight matrices before pdl_wait (lca_grouped_oproj: weights must not be written by work
// still pending on the stream); everything it reads or writes besides them waits.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Round two fp32 values to bf16 (round to nearest even) and pack them (lo in the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Unpack 8 bf16 values held in a 16-byte vector.
__device__ __forceinline__ void unpack8(const uint4 &v, float *f) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float *f) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

// Two fp32 values as fp16 (round to nearest even, saturating at +-65504 instead of overflowing
// to infinity), packed with `first` in the low half.
__device__ __forceinline__ uint32_t pack_f16x2(float first, float second) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(second), "f"(first));
    return r;
}

__device__ __forceinline__ uint4 pack8_f16(const float *f) {
    return make_uint4(pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                      pack_f16x2(f[6], f[7]));
}

// Eight bf16 values re-encoded as fp16.  Exact for magnitudes in [2^-14, 65504] (bf16 carries
// 8 significant bits, fp16 11); smaller ones become fp16 subnormals (absolute error below
// 2^-25), larger ones saturate.
__device__ __forceinline__ uint4 bf16x8_to_f16x8(const uint4 &v) {
    return make_uint4(pack_f16x2(bf16_lo(v.x), bf16_hi(v.x)), pack_f16x2(bf16_lo(v.y), bf16_hi(v.y)),
                      pack_f16x2(bf16_lo(v.z), bf16_hi(v.z)), pack_f16x2(bf16_lo(v.w), bf16_hi(v.w)));
}

// Whether any of the eight bf16 values in v lies outside fp16's finite range: |x| >= 2^16
// (the largest bf16 below that, 65280, is an fp16 value), an infinity or a NaN.
__device__ __forceinline__ bool bf16x8_exceeds_f16(const uint4 &v) {
    const uint32_t mag = 0x7fff7fffu;
    const uint32_t a = __vmaxu2(__vmaxu2(v.x & mag, v.y & mag), __vmaxu2(v.z & mag, v.w & mag));
    return __vcmpgeu2(a, 0x47804780u) != 0;
}

// 2^x by the hardware approximation (relative error about 2^-22; -inf gives 0, results below
// 2^-126 flush to 0): the attention's probabilities, which are then rounded to fp16.
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Sum over the whole block (blockDim.x a multiple of 32, <= 1024); every thread gets it.
__device__ __forceinline__ float block_sum(float v, float *scratch32) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) scratch32[warp] = v;
    __syncthreads();
    float t = lane < nw ? scratch32[lane] : 0.f;
    return warp_sum(t);
}

__device__ __forceinline__ float block_max(float v, float *scratch32) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_max(v);
    __syncthreads();
    if (lane == 0) scratch32[warp] = v;
    __syncthreads();
    float t = lane < nw ? scratch32[lane] : -INFINITY;
    return warp_max(t);
}

// RoPE frequencies as fractions of a turn.  Pair d rotates by pos * theta_d radians with
// theta_d = base^(-2d/R); f[d] = theta_d / (2 pi) in unsigned 0.64 fixed point, computed on
// the host in extended precision.  The angle of position pos is then the 64-bit product
// pos * f[d] taken modulo 2^64 (the whole turns fall off), exact up to the rounding of f[d]
// (~2^-64 relative) even at positions of 2^20 and beyond, with no floating-point range
// reduction on the device.
constexpr int kMaxRopePairs = 64;
struct RopeTable {
    uint64_t f[kMaxRopePairs];
};

// cos/sin of the RoPE angle of pair d at (signed) position pos.
__device__ __forceinline__ void rope_cs(const RopeTable &t, int d, int64_t pos, float &cs, float &sn) {
    const uint64_t turns = (uint64_t)pos * t.f[d];
    const float two_frac = (float)(uint32_t)(turns >> 40) * 0x1p-23f;   // 2 x fraction of a turn
    sincospif(two_frac, &sn, &cs);
}

// e4m3 codes (FP8 caches): round to nearest even, magnitudes past 448 saturate.  hi's code is
// the upper byte of the result, lo's the lower one.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi, float lo) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two e4m3 codes (the first in the low byte) as their exact values.
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t codes, float &first, float &second) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)codes));
    first = __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
    second = __half2float(__ushort_as_half((unsigned short)(h >> 16)));
}

// Two e4m3 codes (the first in the low byte) as an fp16 pair (exact; the first in the low half).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t codes) {
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((uint16_t)codes));
    return h;
}

// An fp16 pair times s2 (both halves), rounded to fp16.
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t x, __half2 s2) {
    __half2 v = *reinterpret_cast<__half2 *>(&x);
    v = __hmul2(v, s2);
    return *reinterpret_cast<uint32_t *>(&v);
}

// The e4m3 codes of f[0..8) / s (IEEE divisions), in memory order; s > 0.
__device__ __forceinline__ uint2 e4m3x8(const float *f, float s) {
    uint32_t w[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const uint32_t lo = cvt_e4m3x2(__fdiv_rn(f[4 * h + 1], s), __fdiv_rn(f[4 * h], s));
        const uint32_t hi = cvt_e4m3x2(__fdiv_rn(f[4 * h + 3], s), __fdiv_rn(f[4 * h + 2], s));
        w[h] = lo | (hi << 16);
    }
    return make_uint2(w[0], w[1]);
}

// Order-preserving map of a float to uint32 (larger float -> larger key); -0 maps like +0.
__device__ __forceinline__ uint32_t ordered_key(float f) {
    if (f == 0.0f) f = 0.0f;
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__host__ __device__ __forceinline__ int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace lca

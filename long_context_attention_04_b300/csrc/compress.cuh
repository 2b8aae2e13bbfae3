// compress.cuh -- KV compression (CSA and HCA) and the sliding-window row writer.
//
// DeepSeek-V4 hybrid attention, CSA step one ("KV 压缩": the KV of every m tokens pooled
// into one entry by a learned, attention-like weighting) and the HCA paragraph (m' tokens
// per entry, no overlap), gxgjx.lffhtl.com/lxrt/355279.html, section 混肃穆力机制; entries
// and window rows are RMS-normalised ("Q/KV normalization") and rotated on their trailing
// dims ("Partial RoPE").
//
// These kernels are bandwidth-trivial (decode reads 2m or m' token rows per sequence);
// one CTA builds one row: softmax weights over the window in shared memory, a 16-byte
// vectorised weighted sum over the tokens, a block reduction for the RMS, the RoPE pairs
// through shared memory, and one coalesced bf16 store.
#pragma once

#include "common.cuh"

namespace lca {

constexpr int kRowThreads = 256;        // threads per window-row CTA
constexpr int kMaxCompressThreads = 1024;  // compressor CTAs: 128..1024 threads, by window size
constexpr int kMaxRowWidth = 1024;      // widest row (elements)
constexpr int kMaxSpan = 256;           // widest compressor window (tokens)

struct RowNormRope {
    const float *gamma;   // [width] or nullptr (no RMSNorm)
    float eps;
    int rope_dims;        // 0: no RoPE
    RopeTable rope;
};

// RMSNorm and RoPE at `pos` of a row held in fp32 shared memory (row[0..width)), in place.
// Every thread of the CTA must call it.
__device__ __forceinline__ void norm_rope_row(float *row, int width, const RowNormRope &nr, int64_t pos,
                                              float *scratch32) {
    if (nr.gamma) {
        float ss = 0.f;
        for (int i = threadIdx.x; i < width; i += blockDim.x) ss += row[i] * row[i];
        ss = block_sum(ss, scratch32);
        const float inv = rsqrtf(ss / (float)width + nr.eps);
        for (int i = threadIdx.x; i < width; i += blockDim.x) row[i] = row[i] * inv * nr.gamma[i];
    }
    __syncthreads();
    if (nr.rope_dims > 0) {
        const int half = nr.rope_dims / 2, base_i = width - nr.rope_dims;
        for (int d = threadIdx.x; d < half; d += blockDim.x) {
            float cs, sn;
            rope_cs(nr.rope, d, pos, cs, sn);
            const float a = row[base_i + d], b = row[base_i + d + half];
            row[base_i + d] = a * cs - b * sn;
            row[base_i + d + half] = a * sn + b * cs;
        }
    }
    __syncthreads();
}

// Finish a row held in fp32 shared memory: RMSNorm, RoPE at `pos`, store bf16.
__device__ __forceinline__ void finish_row(float *row, int width, const RowNormRope &nr, int64_t pos,
                                           __nv_bfloat16 *dst, float *scratch32) {
    norm_rope_row(row, width, nr, pos, scratch32);
    for (int k = threadIdx.x; k < width / 8; k += blockDim.x) {
        reinterpret_cast<uint4 *>(dst)[k] = pack8(row + 8 * k);
    }
}

// Finish a row into an e4m3 cache: RMSNorm and RoPE as above, the row rounded to bf16 (the
// values the bf16 cache would hold), then quantised like quantize_rows_kernel: one fp32
// scale amax / 448 per row, codes e4m3(x / scale).
__device__ __forceinline__ void finish_row_e4m3(float *row, int width, const RowNormRope &nr, int64_t pos,
                                                uint8_t *dst, float *dst_scale, float *scratch32) {
    norm_rope_row(row, width, nr, pos, scratch32);
    float amax = 0.f;
    for (int i = threadIdx.x; i < width; i += blockDim.x) {
        const float b = __bfloat162float(__float2bfloat16_rn(row[i]));
        row[i] = b;
        amax = fmaxf(amax, fabsf(b));
    }
    amax = block_max(amax, scratch32);        // contains __syncthreads: rows visible after it
    const float sc = __fdiv_rn(amax, 448.f);
    if (threadIdx.x == 0) *dst_scale = sc;
    for (int k = threadIdx.x; k < width / 8; k += blockDim.x)
        reinterpret_cast<uint2 *>(dst)[k] = amax > 0.f ? e4m3x8(row + 8 * k, sc) : make_uint2(0u, 0u);
}

struct CompressArgs {
    int span, stride, width;
    const __nv_bfloat16 *tok_v; int64_t tok_v_bs; int n_tok;
    const float *tok_z; int64_t tok_z_bs;
    const int32_t *tok_pos0;
    const float *bias;
    const int32_t *first_entry;
    int n_new;
    __nv_bfloat16 *cache; int64_t cache_bs; int64_t cache_rows;
    RowNormRope nr;
    // e4m3 variant: codes in cache8 (cache_bs and rows in elements = bytes), scales
    uint8_t *cache8;
    float *cache_scale; int64_t scale_bs;
};

// Threads for a compressor CTA: enough that every thread loads about one 16-byte chunk of
// the window (width/8 chunks per token, span tokens), between 128 and 1024.
inline int compress_threads(int width, int span) {
    const int want = (width / 8) * span;
    int t = 128;
    while (t < want && t < kMaxCompressThreads) t *= 2;
    return t;
}

// Dynamic shared memory of a compressor CTA: the token groups' partial sums (two arrays of
// them for per-channel weights: numerators and denominators).
inline size_t compress_smem(int threads, bool per_channel) {
    return (size_t)threads * 8 * sizeof(float) * (per_channel ? 2 : 1);
}

// grid (n_new, batch), block compress_threads(width, span), dynamic shared memory
// compress_smem(threads, PC).
//   PC:  per-channel logits tok_z [n_tok][width] and offset biases bias [span][width], a
//        softmax per channel (the scalar form has one logit per token and one bias per offset).
//   FP8: the entry goes to an e4m3 cache with a per-row scale (finish_row_e4m3).
template <bool PC, bool FP8>
__global__ void __launch_bounds__(kMaxCompressThreads) compress_kernel(CompressArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ float weight[kMaxSpan];
    __shared__ __align__(16) float row[kMaxRowWidth];
    extern __shared__ float partial[];
    __shared__ float scratch[32];
    const int b = blockIdx.y, e = blockIdx.x;
    const int64_t j = (int64_t)a.first_entry[b] + e;
    const int64_t end = (int64_t)a.stride * (j + 1);
    const int64_t nominal = end - a.span;
    const int64_t begin = nominal < 0 ? 0 : nominal;
    const int64_t p0 = a.tok_pos0[b];
    if (j < 0 || j >= a.cache_rows) {
        if (threadIdx.x == 0) raise_error(LCA_DEVERR_VISIBLE_RANGE);
        return;
    }
    if (begin < p0 || end > p0 + a.n_tok) {
        if (threadIdx.x == 0) raise_error(LCA_DEVERR_MISSING_TOKEN);
        return;
    }
    const int n_win = (int)(end - begin);
    const int off0 = (int)(begin - nominal);
    const __nv_bfloat16 *v = a.tok_v + (int64_t)b * a.tok_v_bs + (begin - p0) * a.width;
    const int kc = a.width / 8;                       // 16-byte chunks per row
    const int groups = blockDim.x / kc;               // token groups (>= 1 for width <= 1024)
    const int g = threadIdx.x / kc, k = threadIdx.x % kc;
    if constexpr (PC) {
        // Per channel: thread (group g, chunk k) covers channels 8k .. 8k+7 over the tokens g,
        // g + groups, ...  First the channels' maxima of (z + bias), then exp-weighted sums.
        const float *z = a.tok_z + (int64_t)b * a.tok_z_bs + (begin - p0) * a.width;
        const float *bias = a.bias + (int64_t)off0 * a.width;
        float *pnum = partial;                        // [groups][width]
        float *pden = partial + groups * a.width;     // [groups][width]
        auto logits = [&](int t, float *sv) {
            const float4 *zr = reinterpret_cast<const float4 *>(z + (int64_t)t * a.width + 8 * k);
            const float4 *br = reinterpret_cast<const float4 *>(bias + (int64_t)t * a.width + 8 * k);
            const float4 z0 = __ldg(zr), z1 = __ldg(zr + 1), b0 = __ldg(br), b1 = __ldg(br + 1);
            sv[0] = z0.x + b0.x; sv[1] = z0.y + b0.y; sv[2] = z0.z + b0.z; sv[3] = z0.w + b0.w;
            sv[4] = z1.x + b1.x; sv[5] = z1.y + b1.y; sv[6] = z1.z + b1.z; sv[7] = z1.w + b1.w;
        };
        float mx[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
        if (g < groups) {
            for (int t = g; t < n_win; t += groups) {
                float sv[8];
                logits(t, sv);
#pragma unroll
                for (int u = 0; u < 8; ++u) mx[u] = fmaxf(mx[u], sv[u]);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) pnum[g * a.width + 8 * k + u] = mx[u];
        }
        __syncthreads();
        for (int i = threadIdx.x; i < a.width; i += blockDim.x) {
            float m = -INFINITY;
            for (int gg = 0; gg < groups; ++gg) m = fmaxf(m, pnum[gg * a.width + i]);
            row[i] = m;
        }
        __syncthreads();
        float num[8] = {0, 0, 0, 0, 0, 0, 0, 0}, den[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (g < groups) {
            float cm[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) cm[u] = row[8 * k + u];
            for (int t = g; t < n_win; t += groups) {
                float sv[8], f[8];
                logits(t, sv);
                unpack8(__ldg(reinterpret_cast<const uint4 *>(v + (int64_t)t * a.width) + k), f);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float w = __expf(sv[u] - cm[u]);
                    den[u] += w;
                    num[u] = fmaf(w, f[u], num[u]);
                }
            }
        }
        __syncthreads();                              // every thread has read the maxima
        if (g < groups) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                pnum[g * a.width + 8 * k + u] = num[u];
                pden[g * a.width + 8 * k + u] = den[u];
            }
        }
        __syncthreads();
        for (int i = threadIdx.x; i < a.width; i += blockDim.x) {
            float nsum = 0.f, dsum = 0.f;
            for (int gg = 0; gg < groups; ++gg) {
                nsum += pnum[gg * a.width + i];
                dsum += pden[gg * a.width + i];
            }
            row[i] = nsum / dsum;
        }
    } else {
        const float *z = a.tok_z + (int64_t)b * a.tok_z_bs + (begin - p0);
        // softmax over the surviving tokens of (z_t + bias[offset])
        float mx = -INFINITY;
        for (int t = threadIdx.x; t < n_win; t += blockDim.x) {
            const float s = z[t] + a.bias[off0 + t];
            weight[t] = s;
            mx = fmaxf(mx, s);
        }
        mx = block_max(mx, scratch);
        float den = 0.f;
        for (int t = threadIdx.x; t < n_win; t += blockDim.x) {
            const float w = __expf(weight[t] - mx);
            weight[t] = w;
            den += w;
        }
        den = block_sum(den, scratch);   // contains __syncthreads: weights visible after it
        const float inv_den = 1.f / den;
        // Weighted sum: thread (group g, chunk k) sums 8 channels of chunk k over the tokens
        // g, g + groups, ...; the groups' partial sums are then added in shared memory.
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (g < groups) {
#pragma unroll 4
            for (int t = g; t < n_win; t += groups) {
                const uint4 raw = __ldg(reinterpret_cast<const uint4 *>(v + (int64_t)t * a.width) + k);
                float f[8];
                unpack8(raw, f);
                const float w = weight[t];
#pragma unroll
                for (int u = 0; u < 8; ++u) acc[u] = fmaf(w, f[u], acc[u]);
            }
        }
        float *part = partial;                            // [groups][width]
        if (g < groups) {
#pragma unroll
            for (int u = 0; u < 8; ++u) part[g * a.width + 8 * k + u] = acc[u];
        }
        __syncthreads();
        for (int i = threadIdx.x; i < a.width; i += blockDim.x) {
            float sum = 0.f;
            for (int gg = 0; gg < groups; ++gg) sum += part[gg * a.width + i];
            row[i] = sum * inv_den;
        }
    }
    __syncthreads();
    if constexpr (FP8)
        finish_row_e4m3(row, a.width, a.nr, end - 1, a.cache8 + (int64_t)b * a.cache_bs + j * a.width,
                        a.cache_scale + (int64_t)b * a.scale_bs + j, scratch);
    else
        finish_row(row, a.width, a.nr, end - 1, a.cache + (int64_t)b * a.cache_bs + j * a.width, scratch);
}

struct WindowArgs {
    int width;
    const __nv_bfloat16 *tok_v; int64_t tok_v_bs; int n_tok;
    const int32_t *tok_pos0;
    __nv_bfloat16 *win; int64_t win_bs; int win_cap;
    RowNormRope nr;
};

// grid (n_tok, batch), block kRowThreads: one window row per CTA.
__global__ void __launch_bounds__(kRowThreads) window_kernel(WindowArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ __align__(16) float row[kMaxRowWidth];
    __shared__ float scratch[32];
    const int b = blockIdx.y, t = blockIdx.x;
    const int64_t pos = (int64_t)a.tok_pos0[b] + t;
    if (pos < 0) {
        if (threadIdx.x == 0) raise_error(LCA_DEVERR_NEGATIVE_POS);
        return;
    }
    const __nv_bfloat16 *v = a.tok_v + (int64_t)b * a.tok_v_bs + (int64_t)t * a.width;
    for (int k = threadIdx.x; k < a.width / 8; k += blockDim.x) {
        float f[8];
        unpack8(__ldg(reinterpret_cast<const uint4 *>(v) + k), f);
#pragma unroll
        for (int u = 0; u < 8; ++u) row[8 * k + u] = f[u];
    }
    __syncthreads();
    finish_row(row, a.width, a.nr, pos,
               a.win + (int64_t)b * a.win_bs + (pos % a.win_cap) * a.width, scratch);
}

}  // namespace lca

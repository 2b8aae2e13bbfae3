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

// Finish a row held in fp32 shared memory (row[0..width)): RMSNorm, RoPE at `pos`, store bf16.
// Every thread of the CTA must call it.
__device__ __forceinline__ void finish_row(float *row, int width, const RowNormRope &nr, int64_t pos,
                                           __nv_bfloat16 *dst, float *scratch32) {
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
    for (int k = threadIdx.x; k < width / 8; k += blockDim.x) {
        reinterpret_cast<uint4 *>(dst)[k] = pack8(row + 8 * k);
    }
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
};

// Threads for a compressor CTA: enough that every thread loads about one 16-byte chunk of
// the window (width/8 chunks per token, span tokens), between 128 and 1024.
inline int compress_threads(int width, int span) {
    const int want = (width / 8) * span;
    int t = 128;
    while (t < want && t < kMaxCompressThreads) t *= 2;
    return t;
}

// grid (n_new, batch), block compress_threads(width, span), dynamic shared memory
// blockDim.x * 8 floats (the token groups' partial sums).
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
    const __nv_bfloat16 *v = a.tok_v + (int64_t)b * a.tok_v_bs + (begin - p0) * a.width;
    const int kc = a.width / 8;                       // 16-byte chunks per row
    const int groups = blockDim.x / kc;               // token groups (>= 1 for width <= 1024)
    const int g = threadIdx.x / kc, k = threadIdx.x % kc;
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
    __syncthreads();
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

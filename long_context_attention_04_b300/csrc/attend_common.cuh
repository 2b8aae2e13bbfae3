// attend_common.cuh -- pieces shared by the core-attention kernels: the key-row list of a
// query (compressed rows + window rows), the split of that list across CTAs, the query
// prologue (RMSNorm + RoPE), and the split-K combine with the sink and the output RoPE(-i).
//
// DeepSeek-V4 hybrid attention (gxgjx.lffhtl.com/lxrt/355279.html, section 混肃穆力机制):
// CSA step three (Multi-Query Attention over the top-k compressed blocks), HCA (dense
// attention over all compressed entries), and the tricks list: Q/KV normalization,
// Partial RoPE with the output rotated at -i, the sliding-window branch over the most
// recent uncompressed tokens, and the attention sink in the softmax denominator.
// [P4] zhinnengdao.top section 3.1: one learnable sink logit per head.
#pragma once

#include "common.cuh"

namespace lca {

// Everything an attention kernel needs about one call.
struct AttendArgs {
    int H, C, R;                  // heads, head dim, rope dims
    float eps;
    RopeTable rope;
    float scale_log2;             // softmax scale * log2(e): logits are kept in base 2
    int W;                        // window tokens
    int ratio;                    // m' for the dense (HCA) row list
    int n_idx;                    // k for the gathered (CSA) row list; 0 selects dense
    int n_q;                      // queries per sequence
    int splits;                   // CTAs per query
    const __nv_bfloat16 *q;       // [B][n_q][H][C]
    const float *gamma_q;         // [C]
    const int32_t *q_pos;         // [B][n_q]
    const __nv_bfloat16 *kv; int64_t kv_bs; int64_t cache_rows;
    const float *kv_scale; int64_t ks_bs;   // e4m3 compressed rows (KV8): the rows' scales
    const int32_t *idx;           // [B][n_q][n_idx] or nullptr
    const __nv_bfloat16 *win; int64_t win_bs; int win_cap;
    const float *sink;            // [H]
    // split-K partials: O [unit][split][H][C] fp32 (unnormalised), m/l [unit][split][H] (base 2)
    float *part_o, *part_m, *part_l;
    uint8_t *q_img;               // per-query images of the prepared query: [unit][hi | lo] fp16 (q_prep_kernel)
    __nv_bfloat16 *out;           // [B][n_q][H][C]
    float *lse;                   // [B][n_q][H] or nullptr
};

// The row list of one query: n_comp compressed rows (CSA: idx list, HCA: entries 0..n_vis)
// followed by n_win window rows (tokens win_begin .. pos).
struct RowList {
    int64_t pos;
    int64_t n_comp;
    int64_t win_begin;
    int64_t win_slot0;               // ring row of token win_begin
    int n_win;
    const int32_t *idx;              // CSA list for this query, or nullptr (dense)
    const __nv_bfloat16 *kv;         // this sequence's compressed cache
    const __nv_bfloat16 *win;        // this sequence's window ring
    __device__ __forceinline__ int64_t total() const { return n_comp + n_win; }
};

__device__ __forceinline__ RowList make_row_list(const AttendArgs &a, int b, int qi) {
    RowList L;
    L.pos = a.q_pos[(int64_t)b * a.n_q + qi];
    if (L.pos < 0) {
        raise_error(LCA_DEVERR_NEGATIVE_POS);
        L.pos = -1;
    }
    L.kv = a.kv + (int64_t)b * a.kv_bs;
    L.win = a.win + (int64_t)b * a.win_bs;
    if (a.n_idx > 0) {
        L.idx = a.idx + ((int64_t)b * a.n_q + qi) * a.n_idx;
        L.n_comp = a.n_idx;
    } else {
        L.idx = nullptr;
        int64_t n_vis = (L.pos + 1) / a.ratio;
        if (n_vis > a.cache_rows) {
            raise_error(LCA_DEVERR_VISIBLE_RANGE);
            n_vis = a.cache_rows;
        }
        L.n_comp = n_vis;
    }
    L.win_begin = L.pos - a.W + 1 < 0 ? 0 : L.pos - a.W + 1;
    L.win_slot0 = L.win_begin % a.win_cap;
    L.n_win = (int)(L.pos - L.win_begin + 1);
    return L;
}

// Source of row r of the list, or nullptr when the row is masked (idx == -1 or out of range).
__device__ __forceinline__ const __nv_bfloat16 *row_source(const AttendArgs &a, const RowList &L, int64_t r,
                                                            bool report) {
    if (r < L.n_comp) {
        int64_t j = L.idx ? (int64_t)L.idx[r] : r;
        if (j < 0) return nullptr;
        if (j >= a.cache_rows) {
            if (report) raise_error(LCA_DEVERR_INDEX_RANGE);
            return nullptr;
        }
        return L.kv + j * a.C;
    }
    if (r < L.total()) {
        int64_t slot = L.win_slot0 + (r - L.n_comp);      // at most one wrap: n_win <= W <= win_cap
        if (slot >= a.win_cap) slot -= a.win_cap;
        return L.win + slot * a.C;
    }
    return nullptr;
}

// Query prologue for head h (one warp): RMSNorm over C with gamma_q, then RoPE(pos) on the
// trailing R dims.  Lane l holds elements [l*EPL, l*EPL+EPL) in v[] on return.
// cos/sin of the R/2 RoPE angles at position pos, one pair per thread (threads [0, R/2)).
__device__ __forceinline__ void rope_table_fill(const AttendArgs &a, int64_t pos, float *cs, float *sn) {
    for (int d = threadIdx.x; d < a.R / 2; d += blockDim.x) rope_cs(a.rope, d, pos, cs[d], sn[d]);
}

// One head's query for the calling warp: lane l holds elements [l EPL, l EPL + EPL) of q and
// gamma_q (loaded by q_load_warp, before the position is known, so that the loads overlap).
template <int C>
struct QLane {
    float v[C / 32];
    float g[C / 32];
};

template <int C>
__device__ __forceinline__ void q_load_warp(const AttendArgs &a, const __nv_bfloat16 *qh, QLane<C> &q) {
    constexpr int EPL = C / 32;   // elements per lane (4, 8 or 16)
    const int lane = threadIdx.x & 31;
    if constexpr (EPL >= 8) {
        const uint4 *src = reinterpret_cast<const uint4 *>(qh + lane * EPL);
#pragma unroll
        for (int u = 0; u < EPL / 8; ++u) unpack8(__ldg(src + u), q.v + 8 * u);
    } else {
        const uint2 raw = __ldg(reinterpret_cast<const uint2 *>(qh + lane * EPL));
        q.v[0] = bf16_lo(raw.x); q.v[1] = bf16_hi(raw.x); q.v[2] = bf16_lo(raw.y); q.v[3] = bf16_hi(raw.y);
    }
#pragma unroll
    for (int u = 0; u < EPL; ++u) q.g[u] = __ldg(a.gamma_q + lane * EPL + u);
}

// RMSNorm with gamma_q, then RoPE (table rcs/rsn at the query position) on the trailing R
// dims: the half-split pairs (first + d, first + d + R/2) sit R/2 / EPL lanes apart.
template <int C>
__device__ __forceinline__ void q_hat_warp(const AttendArgs &a, const QLane<C> &q, const float *rcs,
                                           const float *rsn, float *v) {
    constexpr int EPL = C / 32;
    const int lane = threadIdx.x & 31;
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < EPL; ++u) ss += q.v[u] * q.v[u];
    ss = warp_sum(ss);
    const float inv = rsqrtf(ss / (float)C + a.eps);
#pragma unroll
    for (int u = 0; u < EPL; ++u) v[u] = q.v[u] * inv * q.g[u];
    if (a.R > 0) {
        const int half = a.R / 2, first = C - a.R;
        const int hl = half / EPL;        // lanes per half (R/2 is a multiple of EPL)
        const int lane0 = first / EPL;
        const bool in_rope = lane >= lane0;
        const bool lower = lane < lane0 + hl;
        const int partner = lower ? lane + hl : lane - hl;
        // all partner values first, then one branch: the shuffles and the table reads pipeline
        // instead of forming one dependent chain per element
        float other[EPL];
#pragma unroll
        for (int u = 0; u < EPL; ++u) other[u] = __shfl_sync(0xffffffffu, v[u], in_rope ? partner : lane);
        if (in_rope) {
            const int d0 = lane * EPL - first - (lower ? 0 : half);
#pragma unroll
            for (int u = 0; u < EPL; ++u) {
                const float cs = rcs[d0 + u], sn = rsn[d0 + u];
                v[u] = lower ? v[u] * cs - other[u] * sn : other[u] * sn + v[u] * cs;
            }
        }
    }
}

constexpr int kCombineThreads = 128;
constexpr int kMaxSplits = 128;

// Split-K combine: one CTA per (unit, head).  Merges the splits' (m, l, O) with the sink,
// normalises, rotates the trailing R dims by -pos and stores bf16 (+ lse).
//   M = max(sink, max_s m_s);  w_s = 2^(m_s - M);  L = 2^(sink - M) + sum_s w_s l_s;
//   o = sum_s w_s O_s / L   (m, sink in base-2 logit units)
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(AttendArgs a) {
    pdl_trigger();
    pdl_wait();
    __shared__ float wts[kMaxSplits];
    __shared__ __align__(16) float row[1024];
    __shared__ float red[kCombineThreads / 32];
    __shared__ float Lsh;
    const int64_t unit = blockIdx.x;
    const int h = blockIdx.y;
    const int S = a.splits;
    const int64_t pos = a.q_pos[unit] < 0 ? 0 : a.q_pos[unit];
    const float sink2 = a.sink[h] * kLog2e;
    // each thread owns at most one split (S <= kCombineThreads)
    float m = -INFINITY, l = 0.f;
    if (threadIdx.x < S) {
        l = a.part_l[(unit * S + threadIdx.x) * a.H + h];
        m = l > 0.f ? a.part_m[(unit * S + threadIdx.x) * a.H + h] : -INFINITY;
    }
    float M = warp_max(fmaxf(m, sink2));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = M;
    __syncthreads();
    M = red[0];
    for (int w = 1; w < kCombineThreads / 32; ++w) M = fmaxf(M, red[w]);
    const float wgt = threadIdx.x < S && l > 0.f ? exp2f(m - M) : 0.f;
    if (threadIdx.x < S) wts[threadIdx.x] = wgt;
    float part = warp_sum(wgt * l);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = part;
    __syncthreads();
    if (threadIdx.x == 0) {
        float L = exp2f(sink2 - M);
        for (int w = 0; w < kCombineThreads / 32; ++w) L += red[w];
        Lsh = L;
        if (a.lse) a.lse[unit * a.H + h] = (M + log2f(L)) * kLn2;
    }
    __syncthreads();
    const float invL = 1.f / Lsh;
    const float *po = a.part_o + (unit * S * a.H + h) * (int64_t)a.C;
    const int64_t split_stride = (int64_t)a.H * a.C;
    for (int i = 4 * threadIdx.x; i < a.C; i += 4 * blockDim.x) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s2 = 0; s2 < S; ++s2) {
            const float w = wts[s2];
            if (w != 0.f) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(po + s2 * split_stride + i));
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
        }
        row[i] = acc.x * invL;
        row[i + 1] = acc.y * invL;
        row[i + 2] = acc.z * invL;
        row[i + 3] = acc.w * invL;
    }
    __syncthreads();
    if (a.R > 0) {
        const int half = a.R / 2, first = a.C - a.R;
        for (int d = threadIdx.x; d < half; d += blockDim.x) {
            float cs, sn;
            rope_cs(a.rope, d, -pos, cs, sn);
            const float x = row[first + d], y = row[first + d + half];
            row[first + d] = x * cs - y * sn;
            row[first + d + half] = x * sn + y * cs;
        }
    }
    __syncthreads();
    __nv_bfloat16 *dst = a.out + (unit * a.H + h) * a.C;
    for (int k = threadIdx.x; k < a.C / 8; k += blockDim.x)
        reinterpret_cast<uint4 *>(dst)[k] = pack8(row + 8 * k);
}

}  // namespace lca

// attend_simt.cuh -- core attention on the CUDA cores (fp32 FMA), one CTA per
// (query, split).  Writes the same split-K partials as the tensor-core kernel.
#pragma once

#include "attend_common.cuh"

namespace lca {

constexpr int kSimtThreads = 256;
constexpr int kSimtTile = 32;     // rows per tile
constexpr int kSimtHeads = 64;    // head slots (4 threads per head)

template <int C>
struct SimtSmem {
    float q[kSimtHeads][C];
    float kv[kSimtTile][C];
    float p[kSimtHeads][kSimtTile];
    float m[kSimtHeads];
    int valid[kSimtTile];
};

template <int C>
__global__ void __launch_bounds__(kSimtThreads) attend_simt_kernel(AttendArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SimtSmem<C> &sm = *reinterpret_cast<SimtSmem<C> *>(smem_raw);
    constexpr int SEG = C / 4;
    const int unit = blockIdx.x, split = blockIdx.y;
    const int b = unit / a.n_q, qi = unit % a.n_q;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const RowList L = make_row_list(a, b, qi);

    // q prologue: warp w handles heads w, w+8, ...
    for (int h = warp; h < kSimtHeads; h += kSimtThreads / 32) {
        if (h < a.H) {
            float v[C / 32];
            q_hat_warp<C>(a, a.q + ((int64_t)unit * a.H + h) * C, L.pos, v);
#pragma unroll
            for (int u = 0; u < C / 32; ++u) sm.q[h][lane * (C / 32) + u] = v[u];
        } else {
            for (int u = lane; u < C; u += 32) sm.q[h][u] = 0.f;
        }
    }
    const int h = tid >> 2, sub = tid & 3;
    float o[SEG];
#pragma unroll
    for (int u = 0; u < SEG; ++u) o[u] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;

    int64_t t0, t1;
    split_range(L.total(), kSimtTile, split, a.splits, t0, t1);
    for (int64_t t = t0; t < t1; ++t) {
        __syncthreads();
        // load the tile's rows (fp32) and their validity
        for (int r = warp; r < kSimtTile; r += kSimtThreads / 32) {
            const __nv_bfloat16 *src = row_source(a, L, t * kSimtTile + r, lane == 0);
            if (lane == 0) sm.valid[r] = src != nullptr;
            for (int k = lane; k < C / 8; k += 32) {
                float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
                if (src) unpack8(__ldg(reinterpret_cast<const uint4 *>(src) + k), f);
#pragma unroll
                for (int u = 0; u < 8; ++u) sm.kv[r][8 * k + u] = f[u];
            }
        }
        __syncthreads();
        // logits for head h, rows sub + 4i
        float x[kSimtTile / 4];
        float tmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < kSimtTile / 4; ++i) {
            const int r = sub + 4 * i;
            float d = 0.f;
            for (int c = 0; c < C; ++c) d = fmaf(sm.q[h][c], sm.kv[r][c], d);
            x[i] = sm.valid[r] ? d * a.scale_log2 : -INFINITY;
            tmax = fmaxf(tmax, x[i]);
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
        const float m_new = fmaxf(m_run, tmax);
        const float m_use = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = exp2f((m_run == -INFINITY ? m_use : m_run) - m_use);
        float psum = 0.f;
#pragma unroll
        for (int i = 0; i < kSimtTile / 4; ++i) {
            const float p = exp2f(x[i] - m_use);
            sm.p[h][sub + 4 * i] = p;
            psum += p;
        }
        psum += __shfl_xor_sync(0xffffffffu, psum, 1);
        psum += __shfl_xor_sync(0xffffffffu, psum, 2);
        l_run = l_run * alpha + psum;
        m_run = m_new;
#pragma unroll
        for (int u = 0; u < SEG; ++u) o[u] *= alpha;
        __syncthreads();
        for (int r = 0; r < kSimtTile; ++r) {
            const float p = sm.p[h][r];
#pragma unroll
            for (int u = 0; u < SEG; ++u) o[u] = fmaf(p, sm.kv[r][sub * SEG + u], o[u]);
        }
    }
    if (h < a.H) {
        const int64_t pidx = ((int64_t)unit * a.splits + split) * a.H + h;
        float *dst = a.part_o + pidx * C + sub * SEG;
#pragma unroll
        for (int u = 0; u < SEG; ++u) dst[u] = o[u];
        if (sub == 0) {
            a.part_m[pidx] = m_run;
            a.part_l[pidx] = l_run;
        }
    }
}

}  // namespace lca

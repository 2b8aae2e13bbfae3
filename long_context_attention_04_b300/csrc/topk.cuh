// topk.cuh -- exact top-k selection over the indexer scores of each query.
//
// DeepSeek-V4 hybrid attention, CSA step two (gxgjx.lffhtl.com/lxrt/355279.html, section
// 混肃穆力机制: the lightning indexer's scores pick the top-k compressed blocks; "n/m
// becomes top-k"); [P4] section 3.1: top-k = 512 for Flash.
// Order: score descending, index ascending (the lower index wins a tie); output in
// ascending index order, padded with -1 when fewer than k entries are visible.
//
// One CTA per query.  Scores become order-preserving uint32 keys and a three-pass radix
// select (11 + 11 + 10 bits, shared-memory histograms) finds the exact k-th key T and how
// many keys equal to T are needed; a final pass in index order, with one block scan per
// chunk, writes every key > T and the first `need` keys == T, which yields ascending
// indices directly.  Rows of up to kTopkSmemKeys entries (decode) are read from global
// memory once and kept as keys in shared memory for all four passes; longer rows are read
// four times.
#pragma once

#include "common.cuh"

namespace lca {

constexpr int kTopkThreads = 512;
constexpr int kTopkBins = 2048;
constexpr int kTopkSmemKeys = 49152;      // 192 KB of keys in shared memory

struct TopkArgs {
    const float *scores; int64_t row_stride;   // row (b*n_q + i)
    const int32_t *q_pos; int ratio;
    int64_t max_entries;
    int k;
    int32_t *out;                               // [rows][k]
};

// Exclusive prefix sum of one int per thread over the block (kTopkThreads threads).
__device__ __forceinline__ int block_exclusive_scan(int v, int *warp_tot, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    __syncthreads();
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = lane < kTopkThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        if (lane < kTopkThreads / 32) warp_tot[lane] = t;   // inclusive warp totals
    }
    __syncthreads();
    total = warp_tot[kTopkThreads / 32 - 1];
    return x - v + (warp > 0 ? warp_tot[warp - 1] : 0);
}

template <bool SMEM>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(TopkArgs a) {
    extern __shared__ uint32_t skeys[];        // SMEM: the row's keys
    __shared__ int hist[kTopkBins];
    __shared__ int warp_tot[kTopkThreads / 32];
    __shared__ int sel_bin, sel_above;
    const int64_t row = blockIdx.x;
    const float *s = a.scores + row * a.row_stride;
    int32_t *out = a.out + row * (int64_t)a.k;
    const int64_t pos = a.q_pos[row];
    int64_t n = pos < 0 ? 0 : (pos + 1) / a.ratio;
    if (n > a.max_entries) {
        if (threadIdx.x == 0) raise_error(LCA_DEVERR_VISIBLE_RANGE);
        n = a.max_entries;
    }
    const int k = a.k;
    if (n <= k) {
        for (int i = threadIdx.x; i < k; i += blockDim.x) out[i] = i < n ? i : -1;
        return;
    }
    const bool vec4 = ((a.row_stride & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 15) == 0);
    if constexpr (SMEM) {
        const int64_t n4 = vec4 ? n / 4 : 0;
        for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
            const float4 f = __ldg(reinterpret_cast<const float4 *>(s) + i);
            reinterpret_cast<uint4 *>(skeys)[i] =
                make_uint4(ordered_key(f.x), ordered_key(f.y), ordered_key(f.z), ordered_key(f.w));
        }
        for (int64_t i = n4 * 4 + threadIdx.x; i < n; i += blockDim.x) skeys[i] = ordered_key(__ldg(s + i));
        __syncthreads();
    }
    auto key_at = [&](int64_t i) -> uint32_t {
        if constexpr (SMEM) return skeys[i];
        else return ordered_key(__ldg(s + i));
    };
    // ---- radix select of the k-th largest key ----
    uint32_t prefix = 0, mask = 0;
    int remaining = k;     // keys still to take among those matching prefix
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
        const int sh = shifts[pass], nb = 1 << widths[pass];
        for (int i = threadIdx.x; i < nb; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        if (SMEM) {
            for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
                const uint32_t key = skeys[i];
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1)], 1);
            }
        } else if (vec4) {
            const int64_t n4 = n / 4;
            for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
                const float4 f = __ldg(reinterpret_cast<const float4 *>(s) + i);
                const float fv[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const uint32_t key = ordered_key(fv[u]);
                    if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1)], 1);
                }
            }
            for (int64_t i = n4 * 4 + threadIdx.x; i < n; i += blockDim.x) {
                const uint32_t key = ordered_key(__ldg(s + i));
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1)], 1);
            }
        } else {
            for (int64_t i = threadIdx.x; i < n; i += blockDim.x) {
                const uint32_t key = ordered_key(__ldg(s + i));
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> sh) & (nb - 1)], 1);
            }
        }
        __syncthreads();
        // Suffix counts from the top bin down: thread t owns bins nb-1-(q*t .. q*t+q-1).
        const int q = nb / kTopkThreads;   // 4 or 2
        int local = 0;
        for (int u = 0; u < q; ++u) local += hist[nb - 1 - (q * threadIdx.x + u)];
        int total;
        const int before = block_exclusive_scan(local, warp_tot, total);
        // the thread whose range crosses `remaining` finds the bin
        if (before < remaining && before + local >= remaining) {
            int acc = before;
            for (int u = 0; u < q; ++u) {
                const int bin = nb - 1 - (q * threadIdx.x + u);
                const int c = hist[bin];
                if (acc + c >= remaining) {
                    sel_bin = bin;
                    sel_above = acc;
                    break;
                }
                acc += c;
            }
        }
        __syncthreads();
        prefix |= (uint32_t)sel_bin << sh;
        mask |= (uint32_t)(nb - 1) << sh;
        remaining -= sel_above;
        __syncthreads();
    }
    const uint32_t T = prefix;      // the k-th largest key; `remaining` keys equal to T are taken
    // ---- write, in index order: keys > T, and the first `remaining` keys == T ----
    int written = 0, eq_seen = 0;
    for (int64_t base = 0; base < n; base += 4 * kTopkThreads) {
        const int64_t i0 = base + 4 * (int64_t)threadIdx.x;
        uint32_t keys[4];
        int gt = 0, eq = 0;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            keys[u] = i0 + u < n ? key_at(i0 + u) : 0u;
            const bool in = i0 + u < n;
            gt += (in && keys[u] > T);
            eq += (in && keys[u] == T);
        }
        int tot;
        const int packed_before = block_exclusive_scan((gt << 16) | eq, warp_tot, tot);
        int gt_before = packed_before >> 16, eq_before = packed_before & 0xffff;
        int pos_out = written + gt_before + min(max(remaining - eq_seen, 0), eq_before);
        int eq_rank = eq_seen + eq_before;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (i0 + u >= n) break;
            if (keys[u] > T) {
                if (pos_out < k) out[pos_out] = (int32_t)(i0 + u);
                ++pos_out;
            } else if (keys[u] == T) {
                if (eq_rank < remaining) {
                    if (pos_out < k) out[pos_out] = (int32_t)(i0 + u);
                    ++pos_out;
                }
                ++eq_rank;
            }
        }
        const int gt_tot = tot >> 16, eq_tot = tot & 0xffff;
        written += gt_tot + min(max(remaining - eq_seen, 0), eq_tot);
        eq_seen += eq_tot;
        __syncthreads();
    }
}

}  // namespace lca

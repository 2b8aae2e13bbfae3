// topk.cuh -- exact top-k selection over the indexer scores of each query.
//
// DeepSeek-V4 hybrid attention, CSA step two (gxgjx.lffhtl.com/lxrt/355279.html, section
// 混肃穆力机制: the lightning indexer's scores pick the top-k compressed blocks; "n/m
// becomes top-k"); [P4] section 3.1: top-k = 512 for Flash.
// Order: score descending, index ascending (the lower index wins a tie); output in
// ascending index order, padded with -1 when fewer than k entries are visible.
//
// Scores become order-preserving uint32 keys; a three-pass radix select (11 + 11 + 10 bits)
// finds the exact k-th key T and how many keys equal to T are taken (`need`); a last pass
// writes, in index order, every key > T and the first `need` keys == T.
//
// A row is handled by a cluster of `cl` CTAs (1..8; several when there are fewer rows than
// SMs, as in decode), each owning one contiguous slice of the row.  Each CTA builds the
// histogram of its slice in shared memory; the cluster's histograms are summed through
// distributed shared memory, so every CTA picks the same digit.  For the write, each CTA
// counts its slice's outputs, reads the counts of the lower-ranked CTAs, and writes its own
// at the right offset; within a CTA every warp owns a contiguous segment and places its
// outputs with ballots.
//
// After the first digit, each warp keeps, in index order, the keys of its segment whose
// first digit is at or above the selected bin (a few hundred to a few thousand of the row);
// the remaining passes and the write run on those lists only.  Slices of up to
// kTopkSmemKeys entries are read from global memory once and kept as keys in shared memory;
// longer slices (prefill, one CTA per row) are read twice, with 16-byte loads.  If a warp's
// share of the list overflows (heavy ties), the CTA runs the remaining passes over all of
// its keys instead.  When the whole row's lists fit in the first CTA's key area, the other
// CTAs copy theirs there (distributed shared-memory stores, index order kept) and leave, and
// the first CTA runs the remaining passes and the write alone, with no cluster barriers.
#pragma once

#include "common.cuh"

namespace lca {

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkBins = 2048;
constexpr int kTopkMaxCluster = 8;
constexpr int kTopkSmemKeys = 32768;        // 128 KB of keys per CTA in shared memory
constexpr int kTopkCandPerWarp = 256;       // candidate (key, index) pairs per warp: 64 KB in all
constexpr int kTopkUnroll = 8;              // global keys per lane loaded before they are used

__host__ __device__ inline int64_t topk_keys_words(int64_t slice);

struct TopkArgs {
    const float *scores; int64_t row_stride;   // row (b*n_q + i)
    const int32_t *q_pos; int ratio;
    int64_t max_entries;
    int k;
    int cl;                                     // CTAs per row (the cluster size)
    int32_t *out;                               // [rows][k]
};

struct TopkShared {
    int hist[kTopkBins];         // this CTA's histogram
    int merged[kTopkBins];       // the cluster's histogram
    int warp_tot[kTopkWarps];
    int cnt_gt[kTopkWarps], cnt_eq[kTopkWarps];
    int pre_gt[kTopkWarps], pre_eq[kTopkWarps];
    int n_cand[kTopkWarps];
    int cta_gt, cta_eq;          // this CTA's output counts (read by the other CTAs)
    int sel_bin, sel_above, overflow;
    int g_total, g_over;         // this CTA's candidate count and overflow (read by the other CTAs)
};

__device__ __forceinline__ uint32_t smem_u32_of(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster; orders shared-memory writes before the barrier
// with reads after it, across the cluster.
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// Store v to the shared memory of CTA `rank` of the cluster, at the address of `local`.
__device__ __forceinline__ void dsmem_st(const void *local, uint32_t rank, uint32_t v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32_of(local)), "r"(rank));
    asm volatile("st.shared::cluster.b32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

// An int in the shared memory of CTA `rank` of the cluster, at the address of `local`.
// Volatile (kept in program order with the cluster barriers) but without a memory clobber,
// so that several of these loads are in flight before their values are used.
__device__ __forceinline__ int dsmem_ld(const int *local, uint32_t rank) {
    uint32_t remote;
    int v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32_of(local)), "r"(rank));
    asm volatile("ld.shared::cluster.b32 %0, [%1];" : "=r"(v) : "r"(remote));
    return v;
}

// Sum over the cluster's CTAs of the int at `local` (all loads issued before the adds).
__device__ __forceinline__ int dsmem_sum(const int *local, int cl, int upto) {
    int v[kTopkMaxCluster];
#pragma unroll
    for (int r = 0; r < kTopkMaxCluster; ++r) v[r] = r < upto ? dsmem_ld(local, (uint32_t)r) : 0;
    int t = 0;
#pragma unroll
    for (int r = 0; r < kTopkMaxCluster; ++r) t += v[r];
    (void)cl;
    return t;
}

// The digit bin holding the `remaining`-th largest key of `h` (nb bins) and the count of
// keys in the bins above it, written to sh.sel_bin / sh.sel_above.
__device__ __forceinline__ void topk_pick_bin(TopkShared &sh, const int *h, int nb, int remaining) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int q = nb / kTopkThreads;            // 2 or 1 bins per thread, from the top down
    int local = 0;
    for (int u = 0; u < q; ++u) local += h[nb - 1 - (q * threadIdx.x + u)];
    int x = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) sh.warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = sh.warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        sh.warp_tot[lane] = t;
    }
    __syncthreads();
    const int before = x - local + (warp > 0 ? sh.warp_tot[warp - 1] : 0);
    if (before < remaining && before + local >= remaining) {
        int acc = before;
        for (int u = 0; u < q; ++u) {
            const int bin = nb - 1 - (q * threadIdx.x + u);
            const int c = h[bin];
            if (acc + c >= remaining) {
                sh.sel_bin = bin;
                sh.sel_above = acc;
                break;
            }
            acc += c;
        }
    }
    __syncthreads();
}

// Where a CTA's keys come from: keys in shared memory, candidate lists (per warp), or the
// row in global memory.  Keys are addressed by position in the CTA's slice.
struct TopkSrc {
    const uint32_t *skeys;       // [len] shared keys, or nullptr
    const int32_t *sidx;         // [len] row indices of skeys, or nullptr (index = base + position)
    const uint32_t *ckey;        // candidate keys [warps][kTopkCandPerWarp], or nullptr
    const int32_t *cidx;
    const float *g;              // global scores of the slice
    int len;                     // slice length
    int base;                    // row index of slice position 0
    bool vec4;                   // g is 16-byte aligned (float4 loads)
};

// After this CTA's histogram is in sh.hist: the cluster-wide histogram, then the bin.
__device__ __forceinline__ void topk_merge_pick(TopkShared &sh, int cl, int nb, int remaining) {
    if (cl == 1) {
        __syncthreads();
        topk_pick_bin(sh, sh.hist, nb, remaining);
        return;
    }
    cluster_sync();                              // every CTA's histogram is complete
    for (int b = threadIdx.x; b < nb; b += kTopkThreads) sh.merged[b] = dsmem_sum(&sh.hist[b], cl, cl);
    cluster_sync();                              // every CTA is done reading the histograms
    topk_pick_bin(sh, sh.merged, nb, remaining);
}

// Histogram of digit (key >> shift) & (nb-1) over this CTA's keys that match prefix/mask.
__device__ __forceinline__ void topk_hist(TopkShared &sh, const TopkSrc &s, uint32_t prefix, uint32_t mask,
                                          int shift, int nb) {
    for (int i = threadIdx.x; i < nb; i += kTopkThreads) sh.hist[i] = 0;
    __syncthreads();
    const uint32_t dm = (uint32_t)(nb - 1);
    if (s.skeys) {
        for (int i = threadIdx.x; i < s.len; i += kTopkThreads) {
            const uint32_t key = s.skeys[i];
            if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & dm], 1);
        }
    } else if (s.ckey) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        for (int i = lane; i < sh.n_cand[warp]; i += 32) {
            const uint32_t key = s.ckey[warp * kTopkCandPerWarp + i];
            if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & dm], 1);
        }
    } else {
        const int n4 = s.vec4 ? s.len / 4 : 0;
        for (int i0 = threadIdx.x; i0 < n4; i0 += kTopkThreads * kTopkUnroll) {
            float4 f[kTopkUnroll];
#pragma unroll
            for (int u = 0; u < kTopkUnroll; ++u) {      // up to 128 KB of the row in flight per CTA
                const int i = i0 + u * kTopkThreads;
                f[u] = i < n4 ? __ldg(reinterpret_cast<const float4 *>(s.g) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kTopkUnroll; ++u) {
                if (i0 + u * kTopkThreads >= n4) continue;
                const float v[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t key = ordered_key(v[e]);
                    if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & dm], 1);
                }
            }
        }
        for (int i = n4 * 4 + threadIdx.x; i < s.len; i += kTopkThreads) {
            const uint32_t key = ordered_key(__ldg(s.g + i));
            if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & dm], 1);
        }
    }
}

// Key and row index of position i of warp `warp`'s segment (seg keys per warp), valid if in range.
__device__ __forceinline__ uint32_t topk_seg_key(const TopkShared &sh, const TopkSrc &s, int warp, int seg, int i,
                                                 bool &valid, int32_t &index) {
    if (s.ckey) {
        valid = i < sh.n_cand[warp];
        index = valid ? s.cidx[warp * kTopkCandPerWarp + i] : 0;
        return valid ? s.ckey[warp * kTopkCandPerWarp + i] : 0u;
    }
    const int j = warp * seg + i;
    valid = i < seg && j < s.len;
    index = s.sidx ? (valid ? s.sidx[j] : 0) : s.base + j;
    if (!valid) return 0u;
    return s.skeys ? s.skeys[j] : ordered_key(__ldg(s.g + j));
}

// Write, in index order, this CTA's keys > T and its share of the first `need` keys == T.
__device__ __forceinline__ void topk_write(TopkShared &sh, const TopkSrc &s, int cl, uint32_t rank, uint32_t T,
                                           int need, int32_t *out, int k) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int seg = s.ckey ? 0 : ((s.len + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
    const int len = s.ckey ? sh.n_cand[warp] : seg;
    int gt = 0, eq = 0;
    for (int i = lane; i < len; i += 32) {
        bool valid;
        int32_t idx;
        const uint32_t key = topk_seg_key(sh, s, warp, seg, i, valid, idx);
        gt += valid && key > T;
        eq += valid && key == T;
    }
    gt = __reduce_add_sync(0xffffffffu, gt);
    eq = __reduce_add_sync(0xffffffffu, eq);
    if (lane == 0) {
        sh.cnt_gt[warp] = gt;
        sh.cnt_eq[warp] = eq;
    }
    __syncthreads();
    if (warp == 0) {
        const int g0 = sh.cnt_gt[lane], e0 = sh.cnt_eq[lane];
        int a = g0, b = e0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int ya = __shfl_up_sync(0xffffffffu, a, o), yb = __shfl_up_sync(0xffffffffu, b, o);
            if (lane >= o) {
                a += ya;
                b += yb;
            }
        }
        sh.pre_gt[lane] = a - g0;
        sh.pre_eq[lane] = b - e0;
        if (lane == 31) {
            sh.cta_gt = a;
            sh.cta_eq = b;
        }
    }
    // counts of the CTAs before this one in the row
    int gt_before = 0, eq_before = 0;
    if (cl > 1) {
        cluster_sync();
        gt_before = dsmem_sum(&sh.cta_gt, cl, (int)rank);
        eq_before = dsmem_sum(&sh.cta_eq, cl, (int)rank);
    } else {
        __syncthreads();
    }
    int eq_seen = eq_before + sh.pre_eq[warp];                           // keys == T before this point
    int written = gt_before + sh.pre_gt[warp] + min(eq_before + sh.pre_eq[warp], need);
    const uint32_t lt = lanemask_lt();
    for (int i0 = 0; i0 < len; i0 += 32) {
        bool valid;
        int32_t idx;
        const uint32_t key = topk_seg_key(sh, s, warp, seg, i0 + lane, valid, idx);
        const bool is_gt = valid && key > T, is_eq = valid && key == T;
        const uint32_t eq_mask = __ballot_sync(0xffffffffu, is_eq);
        const bool take = is_gt || (is_eq && eq_seen + __popc(eq_mask & lt) < need);
        const uint32_t take_mask = __ballot_sync(0xffffffffu, take);
        if (take) {
            const int o = written + __popc(take_mask & lt);
            if (o < k) out[o] = idx;
        }
        written += __popc(take_mask);
        eq_seen += __popc(eq_mask);
    }
}

// grid (rows * cl), cluster (cl), block kTopkThreads; dynamic shared memory topk_smem_bytes.
template <bool SMEM>
__global__ void __launch_bounds__(kTopkThreads) topk_kernel(TopkArgs a) {
    pdl_trigger();
    pdl_wait();
    extern __shared__ __align__(16) uint32_t dyn[];   // SMEM: slice keys; else candidate keys + indices
    __shared__ TopkShared sh;
    const int cl = a.cl;
    const uint32_t rank = cl > 1 ? cluster_rank() : 0u;
    const int64_t row = blockIdx.x / cl;
    const float *srow = a.scores + row * a.row_stride;
    int32_t *out = a.out + row * (int64_t)a.k;
    const int64_t pos = a.q_pos[row];
    int64_t n64 = pos < 0 ? 0 : (pos + 1) / a.ratio;
    if (n64 > a.max_entries) {
        if (threadIdx.x == 0 && rank == 0) raise_error(LCA_DEVERR_VISIBLE_RANGE);
        n64 = a.max_entries;
    }
    const int n = (int)n64;
    const int k = a.k;
    if (n <= k) {                                // the same decision in every CTA of the row
        if (rank == 0)
            for (int i = threadIdx.x; i < k; i += kTopkThreads) out[i] = i < n ? i : -1;
        return;
    }
    // this CTA's slice of the row, 4-aligned
    const int per = ((n + cl - 1) / cl + 3) & ~3;
    const int lo = min(n, (int)rank * per), hi = min(n, lo + per);
    TopkSrc s{};
    s.g = srow + lo;
    s.len = hi - lo;
    s.base = lo;
    s.vec4 = ((a.row_stride & 3) == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 15) == 0);
    const int cand_off = (int)topk_keys_words(s.len);     // candidates after the keys (SMEM)
    if constexpr (SMEM) {
        const int n4 = s.vec4 ? s.len / 4 : 0;
        for (int i0 = threadIdx.x; i0 < n4; i0 += kTopkUnroll * kTopkThreads) {
            float4 f[kTopkUnroll];
#pragma unroll
            for (int u = 0; u < kTopkUnroll; ++u) {   // up to 128 KB of the row in flight per CTA
                const int i = i0 + u * kTopkThreads;
                f[u] = i < n4 ? __ldg(reinterpret_cast<const float4 *>(s.g) + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kTopkUnroll; ++u) {
                const int i = i0 + u * kTopkThreads;
                if (i < n4)
                    reinterpret_cast<uint4 *>(dyn)[i] = make_uint4(ordered_key(f[u].x), ordered_key(f[u].y),
                                                                   ordered_key(f[u].z), ordered_key(f[u].w));
            }
        }
        for (int i = n4 * 4 + threadIdx.x; i < s.len; i += kTopkThreads) dyn[i] = ordered_key(__ldg(s.g + i));
        __syncthreads();
        s.skeys = dyn;
    }
    int cl_sel = cl;                             // CTAs taking part in the selection from here on
    // ---- first digit (bits 31..21) ----
    topk_hist(sh, s, 0u, 0u, 21, 2048);
    topk_merge_pick(sh, cl, 2048, k);
    const uint32_t bin1 = (uint32_t)sh.sel_bin;
    int remaining = k - sh.sel_above;
    __syncthreads();
    {
        // keep, per warp and in index order, the keys whose first digit is >= bin1: the only
        // keys the rest can select (a few hundred to a few thousand)
        uint32_t *ckey = dyn + (SMEM ? cand_off : 0);
        int32_t *cidx = reinterpret_cast<int32_t *>(ckey + kTopkWarps * kTopkCandPerWarp);
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        const int seg = ((s.len + kTopkWarps - 1) / kTopkWarps + 127) & ~127;
        if (threadIdx.x == 0) sh.overflow = 0;
        __syncthreads();
        int cnt = 0;
        const uint32_t lt = lanemask_lt();
        auto keep_one = [&](uint32_t key, bool in, int j) {
            const bool keep = in && (key >> 21) >= bin1;
            const uint32_t m = __ballot_sync(0xffffffffu, keep);
            if (keep) {
                const int o = cnt + __popc(m & lt);
                if (o < kTopkCandPerWarp) {
                    ckey[warp * kTopkCandPerWarp + o] = key;
                    cidx[warp * kTopkCandPerWarp + o] = s.base + j;
                }
            }
            cnt += __popc(m);
        };
        if (SMEM || !s.vec4) {
            for (int i0 = 0; i0 < seg; i0 += 32) {
                const int j = warp * seg + i0 + lane;
                const bool in = j < s.len;
                const uint32_t key = in ? (SMEM ? s.skeys[j] : ordered_key(__ldg(s.g + j))) : 0u;
                keep_one(key, in, j);
            }
        } else {
            // 128 consecutive keys per step (a float4 per lane), several steps in flight
            for (int i0 = 0; i0 < seg; i0 += 128 * 4) {
                float4 f[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int q = warp * seg + i0 + 128 * u + 4 * lane;
                    f[u] = q + 3 < s.len ? __ldg(reinterpret_cast<const float4 *>(s.g + q))
                                         : make_float4(q < s.len ? __ldg(s.g + q) : 0.f,
                                                       q + 1 < s.len ? __ldg(s.g + q + 1) : 0.f,
                                                       q + 2 < s.len ? __ldg(s.g + q + 2) : 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int q = warp * seg + i0 + 128 * u + 4 * lane;
                    const float v[4] = {f[u].x, f[u].y, f[u].z, f[u].w};
                    uint32_t key[4], bal[4];
                    bool kp[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        key[e] = ordered_key(v[e]);
                        kp[e] = q + e < s.len && (key[e] >> 21) >= bin1;
                        bal[e] = __ballot_sync(0xffffffffu, kp[e]);
                    }
                    int o = cnt;
#pragma unroll
                    for (int e = 0; e < 4; ++e) o += __popc(bal[e] & lt);   // kept keys of lower lanes
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (kp[e]) {
                            if (o < kTopkCandPerWarp) {
                                ckey[warp * kTopkCandPerWarp + o] = key[e];
                                cidx[warp * kTopkCandPerWarp + o] = s.base + q + e;
                            }
                            ++o;
                        }
                        cnt += __popc(bal[e]);
                    }
                }
            }
        }
        if (lane == 0) {
            sh.n_cand[warp] = min(cnt, kTopkCandPerWarp);
            if (cnt > kTopkCandPerWarp) atomicOr(&sh.overflow, 1);
        }
        __syncthreads();
        if (!sh.overflow) {
            s.ckey = ckey;
            s.cidx = cidx;
        }
        // ---- gather: when the whole row's candidates fit in CTA 0's key area, the other CTAs
        // copy theirs there (in index order: CTA by CTA, warp by warp) and leave; CTA 0 finishes
        // the selection alone, with no more cluster barriers.
        if (SMEM && cl > 1) {
            if (warp == 0) {
                const int c = sh.n_cand[lane];
                int x = c;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, x, o);
                    if (lane >= o) x += y;
                }
                sh.pre_gt[lane] = x - c;                 // this warp's offset within the CTA
                if (lane == 31) {
                    sh.g_total = x;
                    sh.g_over = sh.overflow;
                }
            }
            cluster_sync();                              // every CTA's count is readable
            int total = 0, before = 0, over = 0;
            for (int r = 0; r < cl; ++r) {
                const int t = dsmem_ld(&sh.g_total, (uint32_t)r);
                over |= dsmem_ld(&sh.g_over, (uint32_t)r);
                before += r < (int)rank ? t : 0;
                total += t;
            }
            // CTA 0's key area ends where its candidate lists begin (its slice: [0, min(n, per)))
            const int cap = (int)(topk_keys_words(min(n, per)) / 2);    // (key, index) pairs
            if (!over && total <= cap) {
                // CTA 0's key area: keys at [0, cap), indices at [cap, 2 cap)
                const int o0 = before + sh.pre_gt[warp];
                for (int i = lane; i < sh.n_cand[warp]; i += 32) {
                    dsmem_st(dyn + o0 + i, 0u, ckey[warp * kTopkCandPerWarp + i]);
                    dsmem_st(dyn + cap + o0 + i, 0u, (uint32_t)cidx[warp * kTopkCandPerWarp + i]);
                }
                cluster_sync();                          // the copies are in CTA 0
                if (rank != 0) return;
                s.skeys = dyn;
                s.sidx = reinterpret_cast<const int32_t *>(dyn + cap);
                s.ckey = nullptr;
                s.cidx = nullptr;
                s.len = total;
                s.base = 0;
                cl_sel = 1;
            }
        }
    }
    // ---- second and third digits, on keys whose higher digits match ----
    uint32_t prefix = bin1 << 21, mask = 0xFFE00000u;
    topk_hist(sh, s, prefix, mask, 10, 2048);
    topk_merge_pick(sh, cl_sel, 2048, remaining);
    prefix |= (uint32_t)sh.sel_bin << 10;
    mask |= 0x001FFC00u;
    remaining -= sh.sel_above;
    __syncthreads();
    topk_hist(sh, s, prefix, mask, 0, 1024);
    topk_merge_pick(sh, cl_sel, 1024, remaining);
    prefix |= (uint32_t)sh.sel_bin;
    remaining -= sh.sel_above;
    __syncthreads();
    topk_write(sh, s, cl_sel, cl_sel > 1 ? rank : 0u, prefix, remaining, out, k);
    if (cl_sel > 1) cluster_sync();              // keep this CTA's counts readable until all are done
}

// Words of shared memory for a slice's keys, rounded to 16 bytes.
__host__ __device__ inline int64_t topk_keys_words(int64_t slice) { return (slice + 3) & ~(int64_t)3; }

inline size_t topk_smem_bytes(bool smem_keys, int64_t slice) {
    const size_t cand = (size_t)kTopkWarps * kTopkCandPerWarp * 2 * sizeof(uint32_t);
    return (smem_keys ? (size_t)topk_keys_words(slice) * sizeof(uint32_t) : 0) + cand;
}

}  // namespace lca

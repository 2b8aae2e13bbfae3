// topk_stream.cuh -- the top-k of the lightning indexer's scores selected while the scores are
// produced, for prefill chunks (DeepSeek-V4 hybrid attention, gxgjx.lffhtl.com/lxrt/
// 355279.html section 混肃穆力机制, CSA step two: "n/m becomes top-k"; [P4] 3.1).  Order:
// score descending, index ascending (the lower index wins a tie); output in ascending index
// order, padded with -1.
//
// A selection group of 8 indexer epilogue warps (256 threads: the two warp groups, one per
// accumulator buffer, that score the same queries of the current query group) owns those (up
// to kStQueries) queries.  Per query it keeps an append threshold theta (on the order-preserving key of the
// score) and two candidate buffers in global memory (L2-resident workspace), one active.  A
// buffer is a kept region (the survivors of the last compaction) and one append segment per
// warp: a warp appends the scores of its 32 entries whose key is at least theta to its own
// segment, counting in registers (no atomics).  Every kStSyncTiles tiles the warps publish
// their counts; when a segment could overflow before the next check the query is compacted:
// radix passes over the key (11, 11, 10 bits), then over the index for ties, narrow down the
// bin that holds the k-th candidate, and stop as soon as taking that whole bin keeps at most
// 2k candidates.  The kept candidates move to the kept region of the other buffer and theta
// rises to the lowest key that can still enter the top k.  The union property makes this
// exact: every dropped candidate, and every later score below theta, has at least k kept
// candidates above it (a later score whose key equals a kept one has a larger index, so it
// loses that tie).  At the end of the row the same passes select exactly k (stopping early
// only where the selected bin is taken whole), and the k indices are sorted ascending by a
// bitonic sort held in registers (4 per thread; only the strides that cross warps go through
// shared memory).
//
// Every pass reads the buffer with 8 loads in flight per thread.  Synchronisation inside a
// group uses an mbarrier with bounded waits (a wait that runs out raises LCA_DEVERR_TIMEOUT
// and returns false; the caller abandons the row).  Every write into a candidate buffer or the
// sort area is bounds-checked: one that would not fit is dropped and raises LCA_DEVERR_SELECT
// (the counts guarantee it does not happen).
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace lca {

constexpr int kStBins = 2048;
constexpr int kStWarps = 8;              // warps of a selection group (one append segment each)
constexpr int kStQueries = 4;            // queries of a selection group
constexpr int kStThreads = 32 * kStWarps;
constexpr int kStCap = 16384;            // entries of one candidate buffer
constexpr int kStMaxK = 1024;            // largest k of the fused path (also the sort size)
constexpr int kStKeep = 2 * kStMaxK;     // kept region of a buffer (a compaction keeps <= 2k)
constexpr int kStSeg = (kStCap - kStKeep) / kStWarps;    // one warp's append segment (1792)
// tiles between checks: the two sets of a selection group meet only there, so the window is
// long; a set takes every other computed tile of a row, and a warp appends at most 32 a tile
constexpr int kStSyncTiles = 32;
constexpr int kStSegLimit = kStSeg - (kStSyncTiles / 2) * 32;   // a segment past this is compacted
constexpr int kStBatch = 8;              // loads in flight per thread in a pass over a buffer
constexpr int kStPer = kStMaxK / kStThreads;   // sort elements per thread

struct StreamWg {                        // shared state of one selection group
    union {                              // the sort starts after the selection's last radix step
        int hist[kStBins];
        int sort[kStMaxK];
    };
    int part[kStThreads / 32];
    int kept[kStQueries];                // entries in each query's kept region (active buffer)
    int wcnt[kStQueries][kStWarps];      // entries in each warp's segment, as last published
    uint32_t theta[kStQueries];          // append threshold of each query (key >= theta)
    int active[kStQueries];              // which of the query's two buffers is active
    int sel_bin, sel_above, sel_cnt;     // results of a radix step
    int out_cnt;
    uint64_t bar;                        // barrier of the group's warps
};

// The candidates of one query: the kept region of its active buffer (range 0) and the warps'
// segments (ranges 1 .. kStWarps), with their counts as published in shared memory.  (Every
// routine below takes any source with nranges(), range(r) and count(r).)
struct StSrc {
    const uint2 *buf;
    const int *wcnt;
    int kept;
    __device__ __forceinline__ int nranges() const { return 1 + kStWarps; }
    __device__ __forceinline__ int count(int r) const {
        const int c = r == 0 ? kept : wcnt[r - 1];
        const int cap = r == 0 ? kStKeep : kStSeg;   // appends past the end were dropped
        return c < cap ? c : cap;
    }
    __device__ __forceinline__ const uint2 *range(int r) const {
        return buf + (r == 0 ? 0 : kStKeep + (r - 1) * kStSeg);
    }
    __device__ __forceinline__ int total() const {
        int t = 0;
        for (int r = 0; r <= kStWarps; ++r) t += count(r);
        return t;
    }
};

__device__ __forceinline__ uint2 *st_buffer(uint2 *cand, int q, int which) {
    return cand + (int64_t)(q * 2 + which) * kStCap;
}
__device__ __forceinline__ uint2 *st_segment(uint2 *buf, int w) { return buf + kStKeep + w * kStSeg; }

__device__ __forceinline__ StSrc st_source(const StreamWg &s, uint2 *cand, int q) {
    StSrc r;
    r.buf = st_buffer(cand, q, s.active[q]);
    r.wcnt = s.wcnt[q];
    r.kept = s.kept[q];
    return r;
}

// Barrier of the selection group's warps (each warp keeps its own phase count).
__device__ __forceinline__ bool wg_sync(StreamWg &s, uint32_t &phase) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(&s.bar);
    const bool ok = ptx::mbar_wait(&s.bar, phase & 1);
    ++phase;
    return ok;
}

// f(e, valid) for every slot of every range, kStBatch loads issued before any is used; the
// trip counts are the same in every lane (f may use warp collectives).
template <typename Src, typename F>
__device__ __forceinline__ void st_for_each(const Src &src, int tid, F f) {
    const int nr = src.nranges();
#pragma unroll 1
    for (int r = 0; r < nr; ++r) {
        const uint2 *c = src.range(r);
        const int n = src.count(r);
        for (int i0 = 0; i0 < n; i0 += kStBatch * kStThreads) {
            uint2 e[kStBatch];
#pragma unroll
            for (int u = 0; u < kStBatch; ++u) {
                const int i = i0 + u * kStThreads + tid;
                e[u] = i < n ? c[i] : make_uint2(0, 0);
            }
#pragma unroll
            for (int u = 0; u < kStBatch; ++u) f(e[u], i0 + u * kStThreads + tid < n);
        }
    }
}

// One radix step over the candidates: the histogram of digit(e) over the candidates for which
// take(e) holds, then the bin that holds the want-th element (1-based) counted from the top
// bin (desc) or the bottom bin (asc), the number of elements before that bin in that order,
// and the bin's own count: s.sel_bin, s.sel_above, s.sel_cnt.
template <typename Src, typename Take, typename Digit>
__device__ bool wg_radix_step(StreamWg &s, uint32_t &phase, int tid, const Src &src, int nb, int want, bool desc,
                              Take take, Digit digit) {
    for (int b = tid; b < kStBins; b += kStThreads) s.hist[b] = 0;
    if (!wg_sync(s, phase)) return false;
    // every thread has read the previous step's results by now (before arriving at the barrier
    // above): only now may they be reset
    if (tid == 0) {
        s.sel_bin = 0;
        s.sel_above = 0;
        s.sel_cnt = 0;
    }
    st_for_each(src, tid, [&](const uint2 &e, bool valid) {
        if (valid && take(e)) atomicAdd(&s.hist[digit(e)], 1);
    });
    if (!wg_sync(s, phase)) return false;
    // bins in rank order (the order of the selection), nb / 128 per thread
    const int per = (nb + kStThreads - 1) / kStThreads;
    int sum = 0;
    for (int r = tid * per; r < (tid + 1) * per && r < nb; ++r) sum += s.hist[desc ? nb - 1 - r : r];
    const int lane = tid & 31, w = tid >> 5;
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) s.part[w] = incl;
    if (!wg_sync(s, phase)) return false;
    int base = 0;
    for (int k = 0; k < w; ++k) base += s.part[k];
    const int excl = base + incl - sum;
    if (want > excl && want <= excl + sum) {
        int acc = excl;
        for (int r = tid * per; r < (tid + 1) * per && r < nb; ++r) {
            const int bin = desc ? nb - 1 - r : r;
            const int cb = s.hist[bin];
            if (want <= acc + cb) {
                s.sel_bin = bin;
                s.sel_above = acc;
                s.sel_cnt = cb;
                break;
            }
            acc += cb;
        }
    }
    return wg_sync(s, phase);
}

// The candidates taken by a selection: key prefix (kp under mask km) above, or equal and the
// index prefix (ip under mask im) at or below.  A mask of 0 leaves its part undecided.
struct StSel {
    uint32_t kp = 0, km = 0, ip = 0, im = 0;
    __device__ __forceinline__ bool taken(const uint2 &e) const {
        const uint32_t k = e.x & km;
        return k > kp || (k == kp && (e.y & im) <= ip);
    }
    // lowest key a later candidate (a larger index than every one seen) needs to be appended
    __device__ __forceinline__ uint32_t next_theta() const {
        if (km != 0xffffffffu || im == 0) return kp;               // the whole key bin is kept
        return kp == 0xffffffffu ? kp : kp + 1;                     // equal keys lose on index
    }
};

// Narrows the selection of the top `want` (key desc, index asc) of the candidates until the
// candidates taken number at most `limit` (want <= limit; limit == want selects exactly want).
// want <= the number of candidates.  On return *kept is the number of candidates taken.
template <typename Src>
__device__ bool wg_select(StreamWg &s, uint32_t &phase, int tid, const Src &src, int want, int limit, StSel &sel,
                          int &kept) {
    sel = StSel();
    int need = want;                                  // still to take inside the current bin
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    for (int p = 0; p < 6; ++p) {
        const bool key_pass = p < 3;
        const int sh = shifts[p % 3], nb = 1 << widths[p % 3];
        const StSel cur = sel;
        bool ok;
        if (key_pass)
            ok = wg_radix_step(
                s, phase, tid, src, nb, need, true, [&](const uint2 &e) { return (e.x & cur.km) == cur.kp; },
                [&](const uint2 &e) { return (int)((e.x >> sh) & (uint32_t)(nb - 1)); });
        else
            ok = wg_radix_step(
                s, phase, tid, src, nb, need, false,
                [&](const uint2 &e) { return e.x == cur.kp && (e.y & cur.im) == cur.ip; },
                [&](const uint2 &e) { return (int)((e.y >> sh) & (uint32_t)(nb - 1)); });
        if (!ok) return false;
        need -= s.sel_above;
        const uint32_t bin = (uint32_t)s.sel_bin, m = (uint32_t)(nb - 1) << sh;
        if (key_pass) {
            sel.kp |= bin << sh;
            sel.km |= m;
        } else {
            sel.ip |= bin << sh;
            sel.im |= m;
        }
        kept = want - need + s.sel_cnt;               // taking the selected bin whole
        if (kept <= limit) return true;
    }
    return true;                                      // unreachable: the last pass leaves one index
}

// Moves at most 2k of query q's candidates (the top k among them; all of them if there are no
// more than 2k) into the kept region of its other buffer, empties the segments and raises
// theta.  Called by all 128 threads of the group.
__device__ bool wg_compact(StreamWg &s, uint32_t &phase, int tid, uint2 *cand, int q, int k) {
    const StSrc src = st_source(s, cand, q);
    const int n = src.total();
    uint2 *dst = st_buffer(cand, q, s.active[q] ^ 1);
    StSel sel;                                        // km = im = 0: everything taken
    int kept = n;
    if (n > 2 * k && !wg_select(s, phase, tid, src, k, 2 * k, sel, kept)) return false;
    if (tid == 0) s.out_cnt = 0;
    if (!wg_sync(s, phase)) return false;
    st_for_each(src, tid, [&](const uint2 &e, bool valid) {
        const bool take = valid && sel.taken(e);
        const uint32_t m = __ballot_sync(0xffffffffu, take);
        int base = 0;
        if ((tid & 31) == 0 && m) base = atomicAdd(&s.out_cnt, __popc(m));
        base = __shfl_sync(0xffffffffu, base, 0);
        const int pos = base + __popc(m & ((1u << (tid & 31)) - 1u));
        if (take) {
            if (pos < kStKeep) dst[pos] = e;
            else raise_error(LCA_DEVERR_SELECT);
        }
    });
    if (!wg_sync(s, phase)) return false;
    if (tid == 0) {
        s.kept[q] = s.out_cnt < kStKeep ? s.out_cnt : kStKeep;   // == kept
#pragma unroll
        for (int w = 0; w < kStWarps; ++w) s.wcnt[q][w] = 0;
        s.active[q] ^= 1;
        const uint32_t th = sel.next_theta();
        if (th > s.theta[q]) s.theta[q] = th;
    }
    return wg_sync(s, phase);
}

// Compare-exchange of element e (value a) with its partner (value b) at distance `stride`
// inside bitonic blocks of `size`: the lower position of an ascending block keeps the minimum.
__device__ __forceinline__ int bitonic_keep(int e, int a, int b, int size, int stride) {
    const bool up = (e & size) == 0, lo = (e & stride) == 0;
    return (lo == up) ? min(a, b) : max(a, b);
}

// The top k of a source (score descending, index ascending), ascending by index and -1 padded,
// to out[0 .. k) (out may be null).  Called by all threads of the group.
template <typename Src>
__device__ bool wg_select_sorted(StreamWg &s, uint32_t &phase, int tid, const Src &src, int k, int32_t *out) {
    const int n = src.total();
    const int take_n = n < k ? n : k;
    StSel sel;                                        // km = im = 0: everything taken
    int kept = n;
    if (n > k && !wg_select(s, phase, tid, src, k, k, sel, kept)) return false;
    for (int i = tid; i < kStMaxK; i += kStThreads) s.sort[i] = 0x7fffffff;
    if (tid == 0) s.out_cnt = 0;
    if (!wg_sync(s, phase)) return false;
    st_for_each(src, tid, [&](const uint2 &e, bool valid) {
        if (valid && sel.taken(e)) {
            const int pos = atomicAdd(&s.out_cnt, 1);
            if (pos < kStMaxK) s.sort[pos] = (int)e.y;
            else raise_error(LCA_DEVERR_SELECT);
        }
    });
    if (!wg_sync(s, phase)) return false;
    // bitonic sort of kStMaxK indices, ascending (the padding sorts last): thread tid holds
    // elements kStPer tid .. kStPer tid + kStPer - 1; strides below kStPer stay in the thread,
    // strides up to 32 kStPer / 2 are lane shuffles, longer ones go through shared memory
    int v[kStPer];
#pragma unroll
    for (int r = 0; r < kStPer; ++r) v[r] = s.sort[tid * kStPer + r];
    bool fine = true;
#pragma unroll
    for (int size = 2; size <= kStMaxK; size <<= 1) {
#pragma unroll
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            if (stride >= 32 * kStPer) {
                if (!fine) continue;
                fine = wg_sync(s, phase);             // every thread's reads of the last stage are done
#pragma unroll
                for (int r = 0; r < kStPer; ++r) s.sort[tid * kStPer + r] = v[r];
                fine = fine && wg_sync(s, phase);
#pragma unroll
                for (int r = 0; r < kStPer; ++r) {
                    const int e = tid * kStPer + r;
                    v[r] = bitonic_keep(e, v[r], s.sort[e ^ stride], size, stride);
                }
            } else if (stride >= kStPer) {
#pragma unroll
                for (int r = 0; r < kStPer; ++r) {
                    const int b = __shfl_xor_sync(0xffffffffu, v[r], stride / kStPer);
                    v[r] = bitonic_keep(tid * kStPer + r, v[r], b, size, stride);
                }
            } else {
#pragma unroll
                for (int r = 0; r < kStPer; ++r)
                    if ((r & stride) == 0) {
                        const int e = tid * kStPer + r;
                        const int a = v[r], b = v[r | stride];
                        v[r] = bitonic_keep(e, a, b, size, stride);
                        v[r | stride] = bitonic_keep(e | stride, b, a, size, stride);
                    }
            }
        }
    }
    if (!fine) return false;
    if (out) {
#pragma unroll
        for (int r = 0; r < kStPer; ++r) {
            const int i = tid * kStPer + r;
            if (i < k) out[i] = i < take_n ? v[r] : -1;
        }
    }
    return wg_sync(s, phase);
}

// Query q's state back to empty, after its row (or its segment of a row) is done.
__device__ bool wg_reset(StreamWg &s, uint32_t &phase, int tid, int q) {
    if (tid == 0) {
        s.kept[q] = 0;
#pragma unroll
        for (int w = 0; w < kStWarps; ++w) s.wcnt[q][w] = 0;
        s.active[q] = 0;
        s.theta[q] = 0;
    }
    return wg_sync(s, phase);
}

// The final top k of query q, ascending by index and -1 padded, to out[0 .. k) (out may be null:
// the state is reset all the same).
__device__ bool wg_finish(StreamWg &s, uint32_t &phase, int tid, uint2 *cand, int q, int k, int32_t *out) {
    const StSrc src = st_source(s, cand, q);
    return wg_select_sorted(s, phase, tid, src, k, out) && wg_reset(s, phase, tid, q);
}

}  // namespace lca

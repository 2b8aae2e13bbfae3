// attend_tc.cuh -- core attention (CSA and HCA) on the tcgen05 tensor cores.
//
// DeepSeek-V4 hybrid attention (gxgjx.lffhtl.com/lxrt/355279.html, section 混肃穆力机制):
// CSA step three (Multi-Query Attention over the selected compressed blocks), HCA (dense
// attention over every compressed entry), Q/KV normalization, partial RoPE, the sliding-
// window branch and the attention sink; [P4] zhinnengdao.top section 3.1 (c = 512, RoPE on
// the last 64 dims, one sink logit per head).
//
// Multi-Query Attention shares one key/value row set across all heads, so a 128-row tile
// of rows against all (padded to 64) heads is a dense contraction.  Both products run
// transposed so that every MMA has M = 128:
//   S^T[row, head]  = KV[row, c] . Qhat[head, c]^T        (M = 128 rows,  N = 2 x 64, K = c)
//   O^T[c, head]   += KV[row, c]^T . P^T[row, head]       (M = 128 c,     N = 64, K = 128 rows)
// The same 128-byte-swizzled shared-memory tile serves as the K-major A operand of the first
// product and the MN-major A operand of the second.  S^T (128 columns) and O^T (c/128 chunks
// of 64 columns) live in TMEM.
//
// Precision.  Both products run in fp16 with fp32 accumulation.  The KV tile is re-encoded
// in shared memory from bf16 to fp16 as it lands (exact for normalised rows, see
// bf16x8_to_f16x8).  The normalised, rotated query (q_prep_kernel) is split into fp16 hi + lo
// parts (about 22 bits) and S^T accumulates KV.hi^T and KV.lo^T side by side (one N = 128 MMA
// per k step), summed by the softmax: a single fp16 query moves the logits by up to 2^-12 of
// |q||k|, enough to push outputs whose bf16 rounding already sits near the error bound past
// it.  The probabilities, in [0, 1], need no split: fp16 P (relative error 2^-12) lands within
// the output's own bf16 rounding, and the row sum adds the same rounded values.
//
// Shared memory holds the KV tile as four 32 KB slots (128 rows x 128 c each, the whole tile
// at c = 512), a ring of two 32 KB query slots and the 16 KB P^T buffer.  The query is
// not resident: each S chunk comes with the matching 32 KB query chunk (hi and lo stacked as
// one 128-row B operand, bulk-copied from the L2-hot image).  The KV tile stays resident
// across both products; slot j is released when its PV chunk completes, and the producer
// refills it with the next tile's chunk j.  HBM sees one pass over the rows; contiguous tiles
// are prefetched into L2 two tiles ahead.
//
// Rows of a query: compressed rows (CSA: the selected entries; HCA: entries 0..n_vis), then
// the window rows; tiles never mix the two.  All loads are TMA: contiguous compressed tiles
// (HCA) as 2D boxes of 128 rows, indexed rows (CSA selections, window ring rows) with
// 4-row gathers; masked rows are fetched at coordinate -1 and arrive as zeros.
//
// Roles (one CTA per (query, split), one CTA per SM):
//   warp 0      TMA producer of KV chunks
//   warp 10     bulk-copy producer of query chunks
//   warp 11     second issuer of row gathers (c box 1 of gathered chunks; the producer issues
//               box 0): TMA gathers from one warp reach about half the rate of two
//   warp 1      TMEM allocator and MMA issuer (one thread)
//   warps 2-9   re-encoding of each landed KV chunk to fp16 (an eighth each), then the
//               softmax: one TMEM lane (row) per thread, 32 heads per thread; online softmax
//               in base 2 with a conditional rescale (the running max moves only when a
//               logit exceeds it by more than 2^8), P^T rows to shared memory
// The split's unnormalised O, running max and row sum go to the workspace; combine_kernel
// merges the splits with the sink and applies the output RoPE(-pos).
// Every wait is bounded; a wait that runs out raises LCA_DEVERR_TIMEOUT and the CTA unwinds.
#pragma once

#include "attend_common.cuh"
#include "ptx.cuh"
#include "q_prep.cuh"

namespace lca {

constexpr int kAtHP = 64;                                // padded heads (MMA N)
constexpr int kAtTile = 128;                             // rows per tile (MMA M of S^T)
constexpr int kAtSlots = 4;                              // KV chunk slots: one whole tile (c = 512)
constexpr int kAtQSlots = 2;                             // query chunk slots
constexpr int kAtChunkBytes = 128 * 128 * 2;             // KV chunk: 128 rows x 128 c
constexpr int kAtQChunkBytes = kQChunkBytes;             // query chunk: (64 hi + 64 lo) x 128 c
constexpr int kAtProducerWarp = 0;
constexpr int kAtMmaWarp = 1;
constexpr int kAtSoftmaxWarp0 = 2;
constexpr int kAtSoftmaxWarps = 8;
constexpr int kAtQWarp = kAtSoftmaxWarp0 + kAtSoftmaxWarps;
constexpr int kAtGatherWarp = kAtQWarp + 1;              // second issuer of row gathers
constexpr int kAtThreads = 32 * (kAtGatherWarp + 1);
constexpr float kAtTau = 8.0f;                           // log2 headroom before the running max must move

template <int C>
struct AttendTcConfig {
    static constexpr int CC = C / 128;                        // c chunks per row
    static constexpr int P_BYTES = kAtTile * kAtHP * 2;       // fp16 P^T (16 KB)
    static constexpr int TMEM_S = 0;                          // S^T: 128 columns (hi | lo)
    static constexpr int TMEM_O = 2 * kAtHP;                  // O^T chunk j at TMEM_O + 64 j
    static constexpr int TMEM_COLS = 512;
    static constexpr int MISC = 1408;                          // barriers, votes, cross-warp maxima
    static constexpr int SMEM_BYTES = MISC + 1024 + CC * kAtChunkBytes + kAtQSlots * kAtQChunkBytes + P_BYTES;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Where the rows of one query come from, in tiles: tiles [0, tc) hold compressed rows
// [128 t, 128 t + 128) (masked at n_comp), tiles [tc, tc + tw) hold window rows.
struct TileMap {
    int tc, tw;
    __device__ __forceinline__ int total() const { return tc + tw; }
};

__device__ __forceinline__ TileMap tile_map(const RowList &L) {
    TileMap m;
    m.tc = (int)((L.n_comp + kAtTile - 1) / kAtTile);
    m.tw = (L.n_win + kAtTile - 1) / kAtTile;
    return m;
}

// Whether row r of tile t is a real key/value row.
__device__ __forceinline__ bool tile_row_valid(const AttendArgs &a, const RowList &L, const TileMap &m, int t, int r) {
    if (t < m.tc) {
        const int64_t R = (int64_t)t * kAtTile + r;
        if (R >= L.n_comp) return false;
        if (!L.idx) return true;
        const int32_t j = __ldg(L.idx + R);
        return j >= 0 && j < a.cache_rows;
    }
    return (t - m.tc) * kAtTile + r < L.n_win;
}

// Register cap: the register file is split across the four SM sub-partitions (16K each) and
// 11 warps place 3 warps on three of them, so 3 x 32 x 168 <= 16384.
template <int C>
__global__ void __maxnreg__(168) attend_tc_kernel(const __grid_constant__ CUtensorMap kv_tile_map,
                                                  const __grid_constant__ CUtensorMap kv_row_map,
                                                  const __grid_constant__ CUtensorMap win_row_map, AttendArgs a) {
    using Cfg = AttendTcConfig<C>;
    constexpr int CC = Cfg::CC;
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *misc = smem_raw;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw + Cfg::MISC) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *ring = base;                                     // KV slot j = chunk j: 2 boxes [128 rows x 128 B]
    uint8_t *q_ring = ring + CC * kAtChunkBytes;              // query slots: 2 boxes [128 rows x 128 B]
    uint8_t *p_buf = q_ring + kAtQSlots * kAtQChunkBytes;     // P^T: [128 rows x 128 B] fp16
    uint64_t *full = reinterpret_cast<uint64_t *>(misc);
    uint64_t *empty = full + kAtSlots;
    uint64_t *conv = empty + kAtSlots;
    uint64_t *q_full = conv + kAtSlots;
    uint64_t *q_empty = q_full + kAtQSlots;
    uint64_t *s_full = q_empty + kAtQSlots;
    uint64_t *s_empty = s_full + 2;
    uint64_t *p_full = s_empty + 2;
    uint64_t *pv_done = p_full + 2;
    uint64_t *vote_bar = pv_done + 2;
    uint64_t *red_bar = vote_bar + 1;
    uint64_t *teardown = red_bar + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(teardown + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // misc: 27 barriers + TMEM slot + abort flag (224 B), votes, maxima, gather hand-offs
    int *votes = reinterpret_cast<int *>(misc + 256);                  // [2][8]
    float *red = reinterpret_cast<float *>(misc + 320);                // [8][32]
    uint64_t *gather_go = reinterpret_cast<uint64_t *>(misc + 1344);  // [kAtSlots]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // ---- set-up: barriers, TMEM ----
    if (threadIdx.x == 0) {
        for (int s = 0; s < kAtSlots; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
            ptx::mbar_init(&conv[s], kAtSoftmaxWarps);
            ptx::mbar_init(&gather_go[s], 1);
        }
        for (int s = 0; s < kAtQSlots; ++s) {
            ptx::mbar_init(&q_full[s], 1);
            ptx::mbar_init(&q_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&s_full[s], 1);
            ptx::mbar_init(&s_empty[s], kAtSoftmaxWarps);
            ptx::mbar_init(&p_full[s], 32 * kAtSoftmaxWarps);
            ptx::mbar_init(&pv_done[s], 1);
        }
        ptx::mbar_init(vote_bar, kAtSoftmaxWarps);
        ptx::mbar_init(red_bar, kAtSoftmaxWarps);
        ptx::mbar_init(teardown, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == kAtMmaWarp) {
        ptx::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();   // the set-up above touches no global memory; everything below may

    const int unit = blockIdx.x, split = blockIdx.y;
    const int b = unit / a.n_q, qi = unit % a.n_q;
    const RowList L = make_row_list(a, b, qi);
    const TileMap tm = tile_map(L);
    const int64_t t0 = (int64_t)tm.total() * split / a.splits;
    const int64_t t1 = (int64_t)tm.total() * (split + 1) / a.splits;
    const int64_t pidx0 = ((int64_t)unit * a.splits + split) * a.H;
    const uint8_t *qimg = q_img<C>(a, unit);

    if (t0 >= t1) {   // nothing to do for this split: mark it empty for the combine
        for (int h = threadIdx.x; h < a.H; h += blockDim.x) {
            a.part_m[pidx0 + h] = -INFINITY;
            a.part_l[pidx0 + h] = 0.f;
        }
        ptx::tc_fence_before();
        __syncthreads();
        if (warp == kAtMmaWarp) {
            ptx::tc_fence_after();
            ptx::tmem_dealloc(tmem, Cfg::TMEM_COLS);
        }
        return;
    }

    constexpr int kPrefetchTiles = 2;   // contiguous (HCA) tiles are pulled into L2 this far ahead

    const int n_tiles = (int)(t1 - t0);
    const int64_t kv_row0 = (int64_t)b * (a.kv_bs / C);
    const int64_t win_row0 = (int64_t)b * (a.win_bs / C);
    // Rows 4 lane .. 4 lane + 3 of gathered tile t as 2D-map row coordinates (-1: masked, read as 0).
    auto gather_rows = [&](int t, int j, int *rc) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = 4 * lane + i;
            int coord = -1;
            if (t < tm.tc) {
                const int64_t R = (int64_t)t * kAtTile + r;
                if (R < L.n_comp) {
                    const int32_t e = __ldg(L.idx + R);
                    if (e >= 0 && e < a.cache_rows) coord = (int)(kv_row0 + e);
                    else if (e >= a.cache_rows && j == 0 && warp == kAtProducerWarp) raise_error(LCA_DEVERR_INDEX_RANGE);
                }
            } else {
                const int R = (t - tm.tc) * kAtTile + r;
                if (R < L.n_win) {
                    int64_t slot_row = L.win_slot0 + R;   // at most one wrap: n_win <= W <= win_cap
                    if (slot_row >= a.win_cap) slot_row -= a.win_cap;
                    coord = (int)(win_row0 + slot_row);
                }
            }
            rc[i] = coord;
        }
    };

    if (warp == kAtProducerWarp) {
        // ------------------------------------------------------------ producer ----
        // Per tile t: KV chunk j of tile t into slot j, once PV(t-1) has released it.
        if (lane == 0) {
            ptx::tma_prefetch(&kv_tile_map);
            ptx::tma_prefetch(&kv_row_map);
            ptx::tma_prefetch(&win_row_map);
        }
        bool ok = true;
        const int skip = *(volatile int *)&g_test_skip_tile;   // -1 except in the timeout test
        int issued[kAtSlots];                                    // last tile loaded into each slot
        for (int j = 0; j < kAtSlots; ++j) issued[j] = -1;
        for (int u = 0; u < n_tiles && ok && !*abort_flag; ++u) {
            if (u == skip) break;   // test hook: this tile's chunks are never loaded, so their waits run out
            const int t = (int)t0 + u;
            // the tile's gathered rows, once for its c chunks (the index loads overlap the waits)
            int rc[4] = {-1, -1, -1, -1};
            if (t >= tm.tc || L.idx) gather_rows(t, 0, rc);
            for (int j = 0; j < CC && ok; ++j) {
                // KV chunk j of tile t
                if (u > 0 && !ptx::mbar_wait(&empty[j], (u - 1) & 1)) {
                    ok = false;
                    break;
                }
                uint8_t *slot = ring + j * kAtChunkBytes;
                issued[j] = u;
                if (lane == 0) ptx::mbar_arrive_expect_tx(&full[j], kAtChunkBytes);
                __syncwarp();
                const uint32_t dst = ptx::smem_u32(slot);
                if (t < tm.tc && !L.idx) {
                    // contiguous compressed rows: two 64-c boxes of 128 rows
                    if (lane < 2)
                        ptx::tma_load_2d(dst + lane * (128 * 128), &kv_tile_map, j * 128 + lane * 64,
                                         (int)(kv_row0 + (int64_t)t * kAtTile), &full[j]);
                } else {
                    // indexed rows: lane g gathers rows 4g .. 4g+3 of the tile, c box 0; the gather
                    // warp, released through gather_go[j], issues box 1 (one warp's TMA gathers run
                    // at about half the rate of two)
                    if (lane == 0) ptx::mbar_arrive(&gather_go[j]);
                    const CUtensorMap *map = t < tm.tc ? &kv_row_map : &win_row_map;
                    ptx::tma_gather4(dst + lane * 512, map, j * 128, rc[0], rc[1], rc[2], rc[3], &full[j]);
                }
            }
            // L2 prefetch of the next contiguous tiles, issued behind this tile's own loads so that
            // HBM serves those first (at the first tile: the next two)
            if (!L.idx && lane == 1) {
                for (int tp = t + (u == 0 ? 1 : kPrefetchTiles); tp <= t + kPrefetchTiles; ++tp)
                    if (tp < t1 && tp < tm.tc)
                        for (int x = 0; x < C; x += 64)
                            ptx::tma_prefetch_2d(&kv_tile_map, x, (int)(kv_row0 + (int64_t)tp * kAtTile));
            }
        }
        if (!ok) *abort_flag = 1;
        // No copy may still be landing when the CTA exits: wait (bounded) for the last chunk
        // issued into each slot.  Normally the softmax warps have already seen these phases
        // complete, and the waits return at once.  A slot's phase covers the second gather
        // issuer's box as well (its bytes are part of the expected count).
        for (int j = 0; j < kAtSlots; ++j)
            if (issued[j] >= 0) ptx::mbar_wait(&full[j], issued[j] & 1);
    } else if (warp == kAtMmaWarp) {
        // ------------------------------------------------------------- MMA issue ----
        // Per tile: S^T = KV . [hi | lo]^T chunk by chunk as the re-encoded chunks become ready;
        // then, once the softmax has written P,
        // O^T += V^T P^T chunk by chunk, releasing each KV slot to the producer.  tcgen05 ops
        // execute in issue order, so S(t+1) never overwrites S^T or P^T still in use.
        if (lane == 0) {
            constexpr uint32_t idesc_s = ptx::idesc_f16(128, 2 * kAtHP, false, false);
            constexpr uint32_t idesc_o = ptx::idesc_f16(128, kAtHP, true, true);
            const uint32_t p_addr = ptx::smem_u32(p_buf);
            uint32_t q_used = 0;
            bool ok = true;
            for (int u = 0; u < n_tiles && ok && !*abort_flag; ++u) {
                const uint32_t d = tmem + Cfg::TMEM_S;
                for (int j = 0; j < CC && ok; ++j) {
                    const int qs = q_used % kAtQSlots;
                    if (!ptx::mbar_wait(&conv[j], u & 1) || !ptx::mbar_wait(&q_full[qs], (q_used / kAtQSlots) & 1)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t slot = ptx::smem_u32(ring + j * kAtChunkBytes);
                    const uint32_t q_addr = ptx::smem_u32(q_ring + qs * kAtQChunkBytes);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = ptx::smem_desc(slot + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024,
                                                           ptx::kSwizzle128);
                        const uint64_t bd = ptx::smem_desc(q_addr + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024,
                                                           ptx::kSwizzle128);
                        ptx::mma_f16(d, ad, bd, idesc_s, (j > 0 || kk > 0));
                    }
                    ptx::mma_commit(&q_empty[qs]);
                    ++q_used;
                }
                if (!ok) break;
                ptx::mma_commit(&s_full[0]);
                if (!ptx::mbar_wait(&p_full[0], u & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                for (int j = 0; j < CC; ++j) {
                    const uint32_t slot = ptx::smem_u32(ring + j * kAtChunkBytes);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = ptx::smem_desc(slot + kk * 2048, 128 * 128, 1024, ptx::kSwizzle128);
                        const uint64_t bd = ptx::smem_desc(p_addr + kk * 2048, 128 * 128, 1024, ptx::kSwizzle128);
                        ptx::mma_f16(tmem + Cfg::TMEM_O + j * kAtHP, ad, bd, idesc_o, (u > 0 || kk > 0));
                    }
                    ptx::mma_commit(&empty[j]);
                }
                ptx::mma_commit(&pv_done[0]);
            }
            if (!ok) *abort_flag = 1;
            ptx::mma_commit(teardown);
            ptx::mbar_wait(teardown, 0);
        }
    } else if (warp == kAtGatherWarp) {
        // ------------------------------------------------------- second gatherer ----
        // c box 1 of every gathered chunk, after the producer has seen its slot free (gather_go
        // is arrived on once per gathered chunk of the slot, so its phases count those alone).
        uint32_t go_count[kAtSlots] = {};
        bool ok = true;
        for (int u = 0; u < n_tiles && ok && !*abort_flag; ++u) {
            const int t = (int)t0 + u;
            if (t < tm.tc && !L.idx) continue;   // contiguous tile: the producer loads it alone
            int rc[4];
            gather_rows(t, 1, rc);
            for (int j = 0; j < CC; ++j) {
                if (!ptx::mbar_wait(&gather_go[j], go_count[j] & 1)) {
                    ok = false;
                    break;
                }
                ++go_count[j];
                const CUtensorMap *map = t < tm.tc ? &kv_row_map : &win_row_map;
                ptx::tma_gather4(ptx::smem_u32(ring + j * kAtChunkBytes) + 128 * 128 + lane * 512, map,
                                 j * 128 + 64, rc[0], rc[1], rc[2], rc[3], &full[j]);
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == kAtQWarp) {
        // ---------------------------------------------------------- query chunks ----
        // Query chunk j (hi | lo, 32 KB) for every S chunk, in consumption order.
        if (lane == 0) {
            const int total = CC * n_tiles;
            int n = 0;
            for (; n < total && !*abort_flag; ++n) {
                const int qs = n % kAtQSlots, j = n % CC;
                if (n >= kAtQSlots && !ptx::mbar_wait(&q_empty[qs], ((n / kAtQSlots) - 1) & 1)) {
                    *abort_flag = 1;
                    break;
                }
                ptx::mbar_arrive_expect_tx(&q_full[qs], kAtQChunkBytes);
                ptx::bulk_load(ptx::smem_u32(q_ring + qs * kAtQChunkBytes), qimg + j * kAtQChunkBytes, kAtQChunkBytes,
                               &q_full[qs]);
            }
            // the last chunk issued into each slot has landed before the CTA exits (bounded)
            for (int m = n - 1; m >= 0 && m >= n - kAtQSlots; --m)
                ptx::mbar_wait(&q_full[m % kAtQSlots], (m / kAtQSlots) & 1);
        }
    } else {
        // -------------------------------------------------------------- softmax ----
        const int sw = warp - kAtSoftmaxWarp0;       // 0..7
        const int quarter = warp & 3;                // TMEM lane quarter
        const int half = sw >> 2;                    // heads [32 half, 32 half + 32)
        const int r = quarter * 32 + lane;           // row of the tile == TMEM lane
        const uint32_t lane_addr = tmem + ((uint32_t)(quarter * 32) << 16);
        float m[32], l[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
        }
        uint32_t votes_done = 0, reds_done = 0;
        bool ok = true;
        bool range_bad = false;                      // a row element outside fp16's range
        const int ctid = sw * 32 + lane;             // 0..255 among the softmax warps
        for (int u = 0; u < n_tiles && !*abort_flag; ++u) {
            // ---- re-encode tile u's KV chunks to fp16 as they land (an eighth per warp).  The
            // slots were refilled after PV(u-1) released them, which needed this tile's P(u-1).
            for (int j = 0; j < CC && ok; ++j) {
                if (!ptx::mbar_wait(&full[j], u & 1)) {
                    ok = false;
                    break;
                }
                uint4 *chunk = reinterpret_cast<uint4 *>(ring + j * kAtChunkBytes);
#pragma unroll
                for (int k = 0; k < kAtChunkBytes / 16 / (32 * kAtSoftmaxWarps); ++k) {
                    uint4 *p = chunk + ctid + k * (32 * kAtSoftmaxWarps);
                    const uint4 v = *p;
                    range_bad |= bf16x8_exceeds_f16(v);
                    *p = bf16x8_to_f16x8(v);
                }
                ptx::fence_proxy_async();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&conv[j]);
            }
            if (!ok || !ptx::mbar_wait(&s_full[0], u & 1)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            float x[32];
            {
                uint32_t vh[32], vl[32];
                ptx::tmem_ld32(lane_addr + Cfg::TMEM_S + half * 32, vh);
                ptx::tmem_ld32(lane_addr + Cfg::TMEM_S + kAtHP + half * 32, vl);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 32; ++h) x[h] = __uint_as_float(vh[h]) + __uint_as_float(vl[h]);
            }
            ptx::tc_fence_before();
            const bool valid = tile_row_valid(a, L, tm, (int)t0 + u, r);
            bool need = false;
#pragma unroll
            for (int h = 0; h < 32; ++h) {
                x[h] = valid ? x[h] * a.scale_log2 : -INFINITY;
                need |= x[h] > m[h] + kAtTau;
            }
            // ---- CTA-wide vote among the softmax warps: does any running max move? ----
            const int vb = votes_done & 1;
            const bool warp_need = __any_sync(0xffffffffu, need);
            if (lane == 0) votes[vb * 8 + sw] = warp_need ? 1 : 0;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(vote_bar);
            if (!ptx::mbar_wait(vote_bar, votes_done & 1)) {
                ok = false;
                break;
            }
            ++votes_done;
            int any = 0;
#pragma unroll
            for (int w = 0; w < 8; ++w) any |= votes[vb * 8 + w];
            if (any) {
                // Exact per-head maxima of this tile over the 128 rows (4 warps per head half).
                // `red` is single-buffered: every warp has read it before any warp passes the
                // next vote barrier, and only a vote round leads to the next write.
#pragma unroll
                for (int h = 0; h < 32; ++h) {
                    const float mx = warp_max(x[h]);
                    if (lane == h) red[sw * 32 + h] = mx;
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(red_bar);
                if (!ptx::mbar_wait(red_bar, reds_done & 1)) {
                    ok = false;
                    break;
                }
                ++reds_done;
                // O^T: PV of the previous tile completed before S^T of this tile (in-order execution)
#pragma unroll
                for (int h0 = 0; h0 < 32; h0 += 16) {
                    float alpha[16];
                    bool moved = false;
#pragma unroll
                    for (int h = 0; h < 16; ++h) {
                        float mt = m[h0 + h];
#pragma unroll
                        for (int w = 0; w < 4; ++w) mt = fmaxf(mt, red[(half * 4 + w) * 32 + h0 + h]);
                        const float m_old = m[h0 + h] == -INFINITY ? mt : m[h0 + h];
                        alpha[h] = mt == -INFINITY ? 1.f : exp2f(m_old - mt);
                        moved |= alpha[h] != 1.f;
                        m[h0 + h] = mt;
                        l[h0 + h] *= alpha[h];
                    }
                    if (u > 0 && __any_sync(0xffffffffu, moved)) {
#pragma unroll 1
                        for (int j = 0; j < CC; ++j) {
                            uint32_t v[16];
                            const uint32_t addr = lane_addr + Cfg::TMEM_O + j * kAtHP + half * 32 + h0;
                            ptx::tmem_ld16(addr, v);
                            ptx::tmem_ld_wait();
#pragma unroll
                            for (int h = 0; h < 16; ++h) v[h] = __float_as_uint(__uint_as_float(v[h]) * alpha[h]);
                            ptx::tmem_st16(addr, v);
                        }
                        ptx::tmem_st_wait();
                    }
                }
                ptx::tc_fence_before();
            }
            // probabilities of this row as an fp16 P^T row (32 heads = 4 chunks); the row sum
            // adds the rounded values, the weights PV applies.  PV of the previous tile, the last
            // reader of P^T, completed before S^T of this tile.
            float pr[32];
#pragma unroll
            for (int h = 0; h < 32; ++h) {
                const float ms = m[h] == -INFINITY ? 0.f : m[h];
                pr[h] = __half2float(__float2half_rn(exp2f(x[h] - ms)));
                l[h] += pr[h];
            }
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
                *reinterpret_cast<uint4 *>(p_buf + ptx::sw128_offset(r, half * 4 + c4)) = pack8_f16(pr + 8 * c4);
            ptx::fence_proxy_async();
            ptx::mbar_arrive(&p_full[0]);
        }
        if (!ok) *abort_flag = 1;
        // ---- the split's results: row sums, running max, unnormalised O ----
        if (ok && !*abort_flag && ptx::mbar_wait(&pv_done[0], (n_tiles - 1) & 1)) {
            ptx::tc_fence_after();
            // row sums over the 128 rows; the P buffer is free now (every PV is done)
            float *lsum = reinterpret_cast<float *>(p_buf);
#pragma unroll
            for (int h = 0; h < 32; ++h) {
                const float s = warp_sum(l[h]);
                if (lane == h) lsum[sw * 32 + h] = s;
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(red_bar);
            if (ptx::mbar_wait(red_bar, reds_done & 1)) {
                if (quarter == 0) {   // one warp per head half writes m and l
                    const int h = half * 32 + lane;
                    float s = 0.f;
#pragma unroll
                    for (int w = 0; w < 4; ++w) s += lsum[(half * 4 + w) * 32 + lane];
                    float mv = m[0];
#pragma unroll
                    for (int k = 1; k < 32; ++k) mv = lane == k ? m[k] : mv;
                    if (h < a.H) {
                        a.part_m[pidx0 + h] = mv;
                        a.part_l[pidx0 + h] = s;
                    }
                }
                for (int j = 0; j < CC; ++j) {
                    uint32_t v[32];
                    ptx::tmem_ld32(lane_addr + Cfg::TMEM_O + j * kAtHP + half * 32, v);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 32; ++h) {
                        const int hh = half * 32 + h;
                        if (hh < a.H) a.part_o[(pidx0 + hh) * C + j * 128 + r] = __uint_as_float(v[h]);
                    }
                }
            }
            ptx::tc_fence_before();
        }
        if (__any_sync(0xffffffffu, range_bad) && lane == 0) raise_error(LCA_DEVERR_FP16_RANGE);
    }
    __syncthreads();
    if (warp == kAtMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

}  // namespace lca

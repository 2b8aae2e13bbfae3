// attend_tc.cuh -- core attention (CSA and HCA) on the tcgen05 tensor cores.
//
// DeepSeek-V4 hybrid attention (gxgjx.lffhtl.com/lxrt/355279.html, section 混肃穆力机制):
// CSA step three (Multi-Query Attention over the selected compressed blocks), HCA (dense
// attention over every compressed entry), Q/KV normalization, partial RoPE, the sliding-
// window branch and the attention sink; [P4] zhinnengdao.top section 3.1 (c = 512, RoPE on
// the last 64 dims, one sink logit per head).
//
// Multi-Query Attention shares one key/value row set across all heads, so a tile of rows
// against all (padded to 64) heads is a dense contraction.  Per tile of 64 rows:
//   S[q-row, row]   = Qhat[q-row, c] . KV[row, c]^T      (M = 128 query rows, N = 64, K = c)
//   O^T[c, head]   += KV[row, c]^T . P^T[row, head]      (M = 128 c,  N = 64 heads, K = 64)
// The 128 query rows are the 64 heads' normalised, rotated queries split into fp16 hi + lo
// parts (about 22 bits; a single fp16 part moves the logits enough to push outputs whose
// bf16 rounding already sits near the error bound past it).  Query row 32 g + i is the hi
// part of head 16 g + i and row 32 g + 16 + i its lo part, so in S the two parts of a head
// sit in one warp's lane quarter, 16 lanes apart, and a shuffle adds them.
//
// The query is resident for the whole split: its first c - 128 columns in tensor memory (the
// A operand of the logit product read from TMEM), its last 128 columns in shared memory.  That
// leaves shared memory to a ring of ten 16 KB slots of KV chunks (64 rows x 128 c): two and a
// half tiles at c = 512, so the next tiles stream in while a tile's logits, softmax and PV
// run.  Each chunk is re-encoded from bf16 to fp16 in place as it lands (exact for normalised
// rows, see bf16x8_to_f16x8), serves as the K-major B operand of the logit product and then as
// the MN-major A operand of PV, and is released when its PV completes.  The probabilities, in
// [0, 2^8], go to shared memory as fp16 (relative error 2^-12, within the output's own bf16
// rounding), double-buffered so that the softmax of one tile overlaps the PV of the previous.
// TMEM columns: query C - 128 (c >= 256), S 64, O^T c/128 chunks of 64: C in all.
//
// Rows of a query: compressed rows (CSA: the selected entries; HCA: entries 0..n_vis), then
// the window rows; tiles never mix the two.  All loads are TMA: contiguous compressed tiles
// (HCA) as 2D boxes of 64 rows, indexed rows (CSA selections, window ring rows) with 4-row
// gathers; masked rows are fetched at coordinate -1 and arrive as zeros.  A query's tiles are
// cut into contiguous split ranges of equal cost (split_tiles).  The tile height is kAtTile
// (64; the kernel is written for 32 to 64).
//
// Roles (one CTA per (query, split), one CTA per SM, 12 warps; the two MMA issuers sit on
// different SM sub-partitions, warp id mod 4):
//   warp 0      TMA producer of KV chunks (box 0 of gathered chunks, both boxes of contiguous)
//   warp 1      TMEM allocator and issuer of the logit products S (one thread)
//   warp 2      second issuer of row gathers (box 1 of gathered chunks): TMA gathers from one
//               warp reach about half the rate of two
//   warp 3      bulk copy of the prepared query image (q_prep_kernel) into shared memory, then
//               issuer of the PV products (one thread)
//   warps 4-7   softmax, one per TMEM lane quarter: the query's TMEM part at the start, then per
//               tile one head per thread pair (hi lane + lo lane), half the rows each, online
//               base-2 softmax with a conditional rescale (the running max moves only when a logit
//               exceeds it by more than 2^8; the factors go through shared memory so each warp
//               rescales its quarter of O^T), the P row of the head
//   warps 8-11  fp16 re-encoding of each landed KV chunk (a quarter each)
// With KV8 the compressed rows come from an e4m3 cache (one fp32 scale per row; the window
// rows stay bf16): a compressed chunk lands as 64 rows x 128 codes (8 KB, one 128-byte box per
// row) in the upper half of its slot, and the re-encoding warps write fp16(scale x value) into
// the usual fp16 layout over the whole slot (zeros for masked rows): two lanes per row, which
// read the row's codes before either writes (box 1's row covers exactly the row's codes).  Only
// the producer gathers such chunks.
// The split's unnormalised O, running max and row sum go to the workspace; combine_kernel
// merges the splits with the sink and applies the output RoPE(-pos).
// Every wait is bounded; a wait that runs out raises LCA_DEVERR_TIMEOUT and the CTA unwinds
// (issued copies drained, MMAs completed, TMEM freed).
#pragma once

#include "attend_common.cuh"
#include "ptx.cuh"
#include "q_prep.cuh"

namespace lca {

constexpr int kAtHP = 64;                                // padded heads (MMA N of PV)
constexpr int kAtTile = 64;                              // rows per tile (MMA N of the logit product)
constexpr int kAtChunkBytes = kAtTile * 128 * 2;         // KV chunk: kAtTile rows x 128 c
constexpr int kAtBoxBytes = kAtTile * 128;               // one 64-c box of a chunk
constexpr int kAtSlots = (160 * 1024) / kAtChunkBytes;   // KV chunk slots in the ring (160 KB)
constexpr int kAtPBytes = kAtHP * 128;                   // P: 64 heads x kAtTile rows fp16, 128-byte rows (8 KB)
constexpr int kAtRpl = kAtTile / 2;                      // tile rows per softmax lane (hi lane: the first half)
static_assert(kAtTile % 16 == 0 && kAtTile >= 32 && kAtTile <= 64 && kAtRpl % 8 == 0, "tile rows");
static_assert(kAtChunkBytes % 1024 == 0 && kAtBoxBytes % 1024 == 0, "128-byte swizzled boxes start on 1 KB");
constexpr int kAtProducerWarp = 0;
constexpr int kAtMmaWarp = 1;
constexpr int kAtGatherWarp = 2;                         // second issuer of row gathers
constexpr int kAtQWarp = 3;
constexpr int kAtSoftmaxWarp0 = 4;                       // warps 4..7: lane quarters 0..3
constexpr int kAtSoftmaxWarps = 4;
constexpr int kAtConvWarp0 = 8;                          // warps 8..11
constexpr int kAtConvWarps = 4;
constexpr int kAtThreads = 32 * (kAtConvWarp0 + kAtConvWarps);
constexpr float kAtTau = 8.0f;                           // log2 headroom before the running max must move
constexpr int kPrefetchTiles = 2;                        // contiguous (HCA) tiles pulled into L2 this far ahead

template <int C>
struct AttendTcConfig {
    static constexpr int CC = C / 128;                        // c chunks per row
    static constexpr int QT = CC - 1;                         // query chunks held in TMEM
    static constexpr int TMEM_S = QT * 64;                    // S: 64 columns
    static constexpr int TMEM_O = TMEM_S + 64;                // O^T chunk j at TMEM_O + 64 j
    static constexpr int TMEM_COLS = C;
    // ring slots (at its end) that first stage the TMEM query part, image chunk i at offset i x 32 KB
    static constexpr int Q_STAGE_SLOTS = (QT * kQChunkBytes + kAtChunkBytes - 1) / kAtChunkBytes;
    static constexpr int MISC = 2048;                         // barriers, rescale factors, flags
    static constexpr int SMEM_BYTES = MISC + 1024 + kAtSlots * kAtChunkBytes + kQChunkBytes + 2 * kAtPBytes;
    static_assert(TMEM_O + 64 * CC == TMEM_COLS, "tensor memory layout");
    static_assert(Q_STAGE_SLOTS <= kAtSlots - CC, "the first tile and the staged query share the ring");
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Where the rows of one query come from, in tiles: tiles [0, tc) hold compressed rows
// [64 t, 64 t + 64) (masked at n_comp), tiles [tc, tc + tw) hold window rows.
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

// Tiles [t0, t1) of split `split` of `splits`: contiguous ranges of equal cost, where a tile of
// window rows (row gathers) costs kAtWinCost tiles of contiguous compressed rows (2D boxes) in a
// dense (HCA) list (the gathers stream at about half the rate of the boxes, and the window
// tiles all fall to the last split); every tile of a gathered (CSA) list costs one.
constexpr int kAtWinCost = 2;
__device__ __forceinline__ void split_tiles(const TileMap &m, bool gathered, int split, int splits, int64_t &t0,
                                            int64_t &t1) {
    const int64_t w = gathered ? 1 : kAtWinCost;
    const int64_t total = m.tc + w * m.tw;
    auto tile_at = [&](int64_t c) { return c <= m.tc ? c : m.tc + (c - m.tc + w - 1) / w; };
    t0 = tile_at(total * split / splits);
    t1 = tile_at(total * (split + 1) / splits);
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
// 12 warps place 3 on each, so 3 x 32 x 168 <= 16384.
template <int C, bool KV8 = false>
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
    uint8_t *ring = base;                                     // slot s: 2 boxes [kAtTile rows x 128 B]
    uint8_t *q_tail = ring + kAtSlots * kAtChunkBytes;        // last c chunk of the query image (32 KB)
    uint8_t *p_buf = q_tail + kQChunkBytes;                   // 2 x P [64 heads x 128 B] fp16
    uint64_t *full = reinterpret_cast<uint64_t *>(misc);      // chunk landed
    uint64_t *empty = full + kAtSlots;                        // chunk's PV done: slot free
    uint64_t *conv = empty + kAtSlots;                        // chunk re-encoded to fp16
    uint64_t *gather_go = conv + kAtSlots;                    // box 1 may be gathered
    uint64_t *q_full = gather_go + kAtSlots;                  // query image landed
    uint64_t *q_ready = q_full + 1;                           // query's TMEM part written
    uint64_t *q_free = q_ready + 1;                           // staging slots read
    uint64_t *s_full = q_free + 1;
    uint64_t *s_empty = s_full + 1;
    uint64_t *p_full = s_empty + 1;                           // [2]
    uint64_t *pv_done = p_full + 2;                           // [2]
    uint64_t *vote_bar = pv_done + 2;
    uint64_t *teardown = vote_bar + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(teardown + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    // misc: 4 kAtSlots + 11 barriers, TMEM slot, abort flag; rescale factors; their flags
    float *alphas = reinterpret_cast<float *>(misc + 640);    // [2][64]
    int *flags = reinterpret_cast<int *>(misc + 1280);        // [2][4]
    static_assert((4 * kAtSlots + 11) * 8 + 8 <= 640, "barriers fit below the rescale factors");

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // ---- set-up: barriers, TMEM ----
    if (threadIdx.x == 0) {
        for (int s = 0; s < kAtSlots; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
            ptx::mbar_init(&conv[s], kAtConvWarps);
            ptx::mbar_init(&gather_go[s], 1);
        }
        ptx::mbar_init(q_full, 1);
        ptx::mbar_init(q_ready, kAtSoftmaxWarps);
        ptx::mbar_init(q_free, kAtSoftmaxWarps);
        ptx::mbar_init(s_full, 1);
        ptx::mbar_init(s_empty, kAtSoftmaxWarps);
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&p_full[s], kAtSoftmaxWarps);
            ptx::mbar_init(&pv_done[s], 1);
        }
        ptx::mbar_init(vote_bar, kAtSoftmaxWarps);
        ptx::mbar_init(teardown, 2);   // both MMA issuers
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
    int64_t t0, t1;
    split_tiles(tm, L.idx != nullptr, split, a.splits, t0, t1);
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

    const int n_tiles = (int)(t1 - t0);
    const int64_t kv_row0 = (int64_t)b * (a.kv_bs / C);
    const int64_t win_row0 = (int64_t)b * (a.win_bs / C);
    // Rows 4 lane .. 4 lane + 3 (lane < kAtTile / 4) of gathered tile t as 2D-map row coordinates
    // (-1: masked, read as 0).
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
        // Chunk g = u CC + j (tile u, c chunk j) into slot g % kAtSlots once the PV that read the
        // slot's previous chunk has completed; the query's staging slots only after the
        // softmax warps have moved the query to TMEM.
        if (lane == 0) {
            ptx::tma_prefetch(&kv_tile_map);
            ptx::tma_prefetch(&kv_row_map);
            ptx::tma_prefetch(&win_row_map);
        }
        bool ok = true;
        bool staged_free = Cfg::Q_STAGE_SLOTS == 0;
        const int skip = *(volatile int *)&g_test_skip_tile;   // -1 except in the timeout test
        int pf_next = (int)t0 + 1;                               // next tile to prefetch into L2
        int last_g[kAtSlots];                                    // last chunk loaded into each slot
#pragma unroll
        for (int s = 0; s < kAtSlots; ++s) last_g[s] = -1;
        for (int u = 0; u < n_tiles && ok && !*abort_flag; ++u) {
            if (u > 0 && u == skip) break;   // test hook (tile 1 or later): its chunks are never loaded, so
                                             // their waits run out; tile 0's loads never wait for the read
            const int t = (int)t0 + u;
            const bool gathered = t >= tm.tc || L.idx;
            const bool comp8 = KV8 && t < tm.tc;             // e4m3 compressed rows: one 128-code box
            // the tile's gathered rows, once for its c chunks (the index loads overlap the waits)
            int rc[4] = {-1, -1, -1, -1};
            if (gathered && lane < kAtTile / 4) gather_rows(t, 0, rc);
            for (int j = 0; j < CC; ++j) {
                const int g = u * CC + j, slot = g % kAtSlots;
                if (g >= kAtSlots && !ptx::mbar_wait(&empty[slot], ((g / kAtSlots) - 1) & 1)) {
                    ok = false;
                    break;
                }
                if (!staged_free && slot >= kAtSlots - Cfg::Q_STAGE_SLOTS) {
                    if (!ptx::mbar_wait(q_free, 0)) {
                        ok = false;
                        break;
                    }
                    staged_free = true;
                }
#pragma unroll
                for (int s = 0; s < kAtSlots; ++s)
                    if (s == slot) last_g[s] = g;
                const uint32_t dst = ptx::smem_u32(ring + slot * kAtChunkBytes);
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(&full[slot], comp8 ? kAtBoxBytes : kAtChunkBytes);
                    if (gathered && !comp8) ptx::mbar_arrive(&gather_go[slot]);   // box 1 may be gathered now
                }
                __syncwarp();
                if (comp8) {
                    // e4m3 rows into the slot's upper half: 64 contiguous rows, or lane g's 4 gathered rows
                    if (!gathered) {
                        if (lane == 0)
                            ptx::tma_load_2d(dst + kAtBoxBytes, &kv_tile_map, j * 128,
                                             (int)(kv_row0 + (int64_t)t * kAtTile), &full[slot]);
                    } else if (lane < kAtTile / 4) {
                        ptx::tma_gather4(dst + kAtBoxBytes + lane * 512, &kv_row_map, j * 128, rc[0], rc[1], rc[2],
                                         rc[3], &full[slot]);
                    }
                } else if (!gathered) {
                    // contiguous compressed rows: two 64-c boxes of 64 rows
                    if (lane < 2)
                        ptx::tma_load_2d(dst + lane * kAtBoxBytes, &kv_tile_map, j * 128 + lane * 64,
                                         (int)(kv_row0 + (int64_t)t * kAtTile), &full[slot]);
                } else if (lane < kAtTile / 4) {
                    // indexed rows: lane g gathers rows 4g .. 4g+3 of the tile, c box 0
                    const CUtensorMap *map = t < tm.tc ? &kv_row_map : &win_row_map;
                    ptx::tma_gather4(dst + lane * 512, map, j * 128, rc[0], rc[1], rc[2], rc[3], &full[slot]);
                }
            }
            // L2 prefetch of contiguous tiles ahead, issued behind this tile's own loads; the
            // distance ramps up over the first tiles, so that at launch, when every CTA loads at
            // once, the tiles needed first are not queued behind tiles needed later
            if (ok && !L.idx && lane == 1) {
                const int target = t + (u < kPrefetchTiles ? u + 1 : kPrefetchTiles);
                for (; pf_next <= target; ++pf_next)
                    if (pf_next < t1 && pf_next < tm.tc)
                        for (int x = 0; x < C; x += (KV8 ? 128 : 64))
                            ptx::tma_prefetch_2d(&kv_tile_map, x, (int)(kv_row0 + (int64_t)pf_next * kAtTile));
            }
        }
        if (!ok) *abort_flag = 1;
        // No copy may still be landing when the CTA exits: wait (bounded) for the last chunk
        // issued into each slot.  Normally the conversion warps have already seen these phases
        // complete, and the waits return at once.  A slot's phase covers the second gather
        // issuer's box as well (its bytes are part of the expected count).
#pragma unroll
        for (int s = 0; s < kAtSlots; ++s)
            if (last_g[s] >= 0) ptx::mbar_wait(&full[s], (last_g[s] / kAtSlots) & 1);
    } else if (warp == kAtGatherWarp) {
        // ------------------------------------------------------- second gatherer ----
        // c box 1 of every gathered chunk, after the producer has claimed the chunk's slot.  The
        // gathered tiles are all of them (CSA) or the trailing window tiles (HCA), so with gfirst
        // the first gathered chunk, gathered chunk g is the ((g - gfirst) / kAtSlots)-th to use
        // its slot's go barrier.
        bool ok = true;
        const int u_first = (L.idx && !KV8) ? 0 : (int)(tm.tc > t0 ? tm.tc - t0 : 0);
        const int gfirst = u_first * CC;
        for (int u = u_first; u < n_tiles && ok && !*abort_flag; ++u) {
            const int t = (int)t0 + u;
            int rc[4] = {-1, -1, -1, -1};
            if (lane < kAtTile / 4) gather_rows(t, 1, rc);
            for (int j = 0; j < CC; ++j) {
                const int g = u * CC + j, slot = g % kAtSlots;
                if (!ptx::mbar_wait(&gather_go[slot], ((g - gfirst) / kAtSlots) & 1)) {
                    ok = false;
                    break;
                }
                if (lane < kAtTile / 4) {
                    const CUtensorMap *map = t < tm.tc ? &kv_row_map : &win_row_map;
                    ptx::tma_gather4(ptx::smem_u32(ring + slot * kAtChunkBytes) + kAtBoxBytes + lane * 512, map,
                                     j * 128 + 64, rc[0], rc[1], rc[2], rc[3], &full[slot]);
                }
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == kAtQWarp) {
        // ---------------------------------------------------- query image, then PV ----
        // Chunks 0 .. CC-2 into the staging slots (the softmax warps move them to TMEM), the last
        // chunk into its own area (the smem A operand of the last k steps).  Then this warp's
        // lane 0 issues every PV product: PV(v) as soon as P(v) is written, independently of the
        // logit products, which warp 1 issues on another SM sub-partition (one issuing thread
        // for both lost about half its issue rate to the other warps of its sub-partition).
        if (lane == 0) {
            ptx::mbar_arrive_expect_tx(q_full, CC * kQChunkBytes);
            for (int i = 0; i < CC - 1; ++i)
                ptx::bulk_load(ptx::smem_u32(ring + (kAtSlots - Cfg::Q_STAGE_SLOTS) * kAtChunkBytes + i * kQChunkBytes),
                               qimg + i * kQChunkBytes, kQChunkBytes, q_full);
            ptx::bulk_load(ptx::smem_u32(q_tail), qimg + (CC - 1) * kQChunkBytes, kQChunkBytes, q_full);
            bool ok = ptx::mbar_wait(q_full, 0);   // landed before the CTA can exit
            constexpr uint32_t idesc_o = ptx::idesc_f16(128, kAtHP, true, false);
            const uint64_t kv_mn = ptx::smem_desc(ptx::smem_u32(ring), kAtBoxBytes, 1024, ptx::kSwizzle128);  // MN-major A
            const uint64_t p_k = ptx::smem_desc(ptx::smem_u32(p_buf), 16, 1024, ptx::kSwizzle128);
            for (int v = 0; v < n_tiles && ok && !*abort_flag; ++v) {
                if (!ptx::mbar_wait(&p_full[v & 1], (v >> 1) & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint64_t pb = p_k + (uint64_t)((v & 1) * (kAtPBytes >> 4));
                const uint32_t first = v > 0 ? 1u : 0u;
#pragma unroll
                for (int j = 0; j < CC; ++j) {
                    const int g = v * CC + j, slot = g % kAtSlots;
                    const uint64_t ad0 = kv_mn + (uint64_t)(slot * (kAtChunkBytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < kAtTile / 16; ++kk)
                        ptx::mma_f16(tmem + Cfg::TMEM_O + j * 64, ad0 + kk * (2048 >> 4), pb + kk * 2, idesc_o,
                                     kk > 0 ? 1u : first);
                    ptx::mma_commit(&empty[slot]);   // the slot's S product completed before P(v) existed
                }
                ptx::mma_commit(&pv_done[v & 1]);
            }
            if (!ok) *abort_flag = 1;
            ptx::mma_commit(teardown);
            ptx::mbar_wait(teardown, 0);
        }
    } else if (warp >= kAtConvWarp0) {
        // ------------------------------------------------------ fp16 re-encoding ----
        const int ct = (warp - kAtConvWarp0) * 32 + lane;   // 0 .. 127
        bool ok = true, range_bad = false;
        const int total = n_tiles * CC;
        // KV8: lanes 2r and 2r + 1 own row r of a compressed chunk (codes 0..63 and 64..127); the
        // row's scale (0 for a masked row) is loaded a tile ahead, off the chunk's path
        const int crow = ct >> 1, chalf = ct & 1;
        const float *kscale = KV8 ? a.kv_scale + (int64_t)b * a.ks_bs : nullptr;
        auto load_scale = [&](int u) -> float {
            const int64_t t = t0 + u;
            if (!KV8 || u >= n_tiles || t >= tm.tc || crow >= kAtTile) return 0.f;
            const int64_t R = t * kAtTile + crow;
            if (R >= L.n_comp) return 0.f;
            int64_t e = R;
            if (L.idx) {
                e = __ldg(L.idx + R);
                if (e < 0 || e >= a.cache_rows) return 0.f;
            }
            return __ldg(kscale + e);
        };
        float sc_cur = 0.f, sc_next = KV8 ? load_scale(0) : 0.f;
        for (int g = 0; g < total && !*abort_flag; ++g) {
            const int slot = g % kAtSlots;
            const int u = g / CC;
            if (KV8 && g % CC == 0) {
                sc_cur = sc_next;
                sc_next = load_scale(u + 1);
            }
            if (!ptx::mbar_wait(&full[slot], (g / kAtSlots) & 1)) {
                ok = false;
                break;
            }
            uint8_t *sl = ring + slot * kAtChunkBytes;
            if (KV8 && t0 + u < tm.tc) {
                // e4m3 chunk: the row's codes sit in the slot's upper half (swizzled 128-byte rows);
                // its fp16 values go to box 0 (codes 0..63, this row's lane 2r) and box 1 (codes
                // 64..127, lane 2r + 1), and box 1's row covers exactly this row's codes: both lanes
                // read first, then write
                const int r = crow;
                const bool has_row = kAtTile == 64 || r < kAtTile;   // lanes past the tile's rows idle
                uint4 e[4] = {};
                if (has_row)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int u8 = 4 * chalf + i;
                        e[i] = *reinterpret_cast<const uint4 *>(sl + kAtBoxBytes + r * 128 + ((u8 ^ (r & 7)) << 4));
                    }
                __syncwarp();
                // fp16(value) x fp16(scale), rounded to fp16 (about 2^-10 relative, inside the codes'
                // own 2^-4); the largest e4m3 magnitude, 448, times the scale must fit fp16, and a
                // NaN code of a row that is read is reported (masked rows, scale 0, become zeros)
                const float s = sc_cur;
                const bool live = s > 0.f;
                const __half2 s2 = __float2half2_rn(s);
                range_bad |= live && !(s * 448.f <= 65504.f);
                uint8_t *row = sl + chalf * kAtBoxBytes + r * 128;
#pragma unroll
                for (int i = 0; i < 4 && has_row; ++i) {
                    const uint32_t words[4] = {e[i].x, e[i].y, e[i].z, e[i].w};
                    uint32_t w[8];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        range_bad |= live && __vcmpeq4(words[q] & 0x7f7f7f7fu, 0x7f7f7f7fu) != 0;
                        w[2 * q] = live ? hmul2_u32(e4m3x2_to_f16x2(words[q] & 0xffffu), s2) : 0u;
                        w[2 * q + 1] = live ? hmul2_u32(e4m3x2_to_f16x2(words[q] >> 16), s2) : 0u;
                    }
                    const int v0 = 2 * i;
                    *reinterpret_cast<uint4 *>(row + ((v0 ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    *reinterpret_cast<uint4 *>(row + (((v0 + 1) ^ (r & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
                }
            } else {
                uint4 *chunk = reinterpret_cast<uint4 *>(sl);
#pragma unroll
                for (int k = 0; k < kAtChunkBytes / 16 / (32 * kAtConvWarps); ++k) {
                    uint4 *p = chunk + ct + k * (32 * kAtConvWarps);
                    const uint4 v = *p;
                    range_bad |= bf16x8_exceeds_f16(v);
                    *p = bf16x8_to_f16x8(v);
                }
            }
            ptx::fence_proxy_async();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&conv[slot]);
        }
        if (!ok) *abort_flag = 1;
        if (__any_sync(0xffffffffu, range_bad) && lane == 0) raise_error(LCA_DEVERR_FP16_RANGE);
    } else if (warp == kAtMmaWarp) {
        // ------------------------------------------------------------- S issue ----
        // S(u) chunk by chunk as the re-encoded chunks become ready, once the softmax has read
        // S(u-1) out of tensor memory; PV is issued by warp 3.  Each issuer commits its own
        // products (tcgen05.commit tracks the issuing thread's operations).
        if (lane == 0) {
            constexpr uint32_t idesc_s = ptx::idesc_f16(128, kAtTile, false, false);
            // Matrix descriptors computed once: a byte offset o inside shared memory moves the
            // descriptor's start-address field by o / 16, so every operand below is a base
            // descriptor plus a constant (the issue loop must stay faster than the tensor pipe).
            const uint64_t kv_k = ptx::smem_desc(ptx::smem_u32(ring), 16, 1024, ptx::kSwizzle128);   // K-major B
            const uint64_t qt_k = ptx::smem_desc(ptx::smem_u32(q_tail), 16, 1024, ptx::kSwizzle128);
            const uint32_t d_s = tmem + Cfg::TMEM_S;
            bool ok = ptx::mbar_wait(q_ready, 0);
            ptx::tc_fence_after();
            for (int u = 0; u < n_tiles && ok && !*abort_flag; ++u) {
                if (u > 0 && !ptx::mbar_wait(s_empty, (u - 1) & 1)) {
                    ok = false;
                    break;
                }
                for (int jc = 0; jc < CC; ++jc) {
                    const int g = u * CC + jc, slot = g % kAtSlots;
                    if (!ptx::mbar_wait(&conv[slot], (g / kAtSlots) & 1)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t bd0 = kv_k + (uint64_t)(slot * (kAtChunkBytes >> 4));
                    if (jc < CC - 1) {
                        const uint32_t a0 = tmem + jc * 64;
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            ptx::mma_f16_ts(d_s, a0 + kk * 8, bd0 + ((kk >> 2) * (kAtBoxBytes >> 4) + (kk & 3) * 2),
                                            idesc_s, (jc > 0 || kk > 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            ptx::mma_f16(d_s, qt_k + ((kk >> 2) * ((128 * 128) >> 4) + (kk & 3) * 2),
                                         bd0 + ((kk >> 2) * (kAtBoxBytes >> 4) + (kk & 3) * 2), idesc_s,
                                         (CC > 1 || kk > 0) ? 1u : 0u);
                    }
                }
                if (!ok) break;
                ptx::mma_commit(s_full);
            }
            if (!ok) *abort_flag = 1;
            ptx::mma_commit(teardown);
            ptx::mbar_wait(teardown, 0);
        }
    } else {
        // -------------------------------------------------------------- softmax ----
        // Warp q (lane quarter q) owns query rows 32 q .. 32 q + 31: lane l < 16 the hi part of
        // head 16 q + l, lane l + 16 its lo part.  Per tile the hi lane takes the first kAtRpl tile
        // rows of its head and the lo lane the other kAtRpl, each adding the partner's part.
        const int q = warp & 3;
        const int part = lane >> 4;
        const int h = 16 * q + (lane & 15);
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        bool ok = ptx::mbar_wait(q_full, 0);
        if (ok) {
            // the query's TMEM part: this lane's row of image chunks 0 .. CC-2
            const int row = 32 * q + lane;
            for (int i = 0; i < CC - 1; ++i) {
                const uint8_t *img = ring + (kAtSlots - Cfg::Q_STAGE_SLOTS) * kAtChunkBytes + i * kQChunkBytes;
                uint32_t v[64];
#pragma unroll
                for (int bx = 0; bx < 2; ++bx)
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(img + bx * (128 * 128) + sw128(row, k));
                        v[bx * 32 + 4 * k + 0] = w.x;
                        v[bx * 32 + 4 * k + 1] = w.y;
                        v[bx * 32 + 4 * k + 2] = w.z;
                        v[bx * 32 + 4 * k + 3] = w.w;
                    }
                ptx::tmem_st32(lane_base + i * 64, v);
                ptx::tmem_st32(lane_base + i * 64 + 32, v + 32);
            }
            ptx::tmem_st_wait();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
            ptx::mbar_arrive(q_ready);
            ptx::mbar_arrive(q_free);
        }
        float m_run = -INFINITY, l_run = 0.f;
        for (int u = 0; u < n_tiles && ok && !*abort_flag; ++u) {
            const int t = (int)t0 + u;
            if (!ptx::mbar_wait(s_full, u & 1)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            float x[kAtRpl];
            {
                uint32_t sv[kAtTile];
                ptx::tmem_ld32(lane_base + Cfg::TMEM_S, sv);
                if constexpr (kAtTile == 64) ptx::tmem_ld32(lane_base + Cfg::TMEM_S + 32, sv + 32);
                else if constexpr (kAtTile == 48) ptx::tmem_ld16(lane_base + Cfg::TMEM_S + 32, sv + 32);
                ptx::tmem_ld_wait();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(s_empty);   // S may be overwritten by the next tile
                // row validity of the tile's rows (64-bit: bit r for row r), this lane's half
                const uint32_t m0 = __ballot_sync(0xffffffffu, tile_row_valid(a, L, tm, t, lane));
                const uint32_t m1 = kAtTile > 32 ? __ballot_sync(0xffffffffu, tile_row_valid(a, L, tm, t, lane + 32)) : 0u;
                const uint32_t mask = (uint32_t)((((uint64_t)m1 << 32) | m0) >> (part * kAtRpl));
#pragma unroll
                for (int i = 0; i < kAtRpl; ++i) {
                    // hi lane: own hi[i] + partner's lo[i]; lo lane: own lo[R+i] + partner's hi[R+i]
                    const float send = __uint_as_float(part ? sv[i] : sv[kAtRpl + i]);
                    const float mine = __uint_as_float(part ? sv[kAtRpl + i] : sv[i]);
                    const float other = __shfl_xor_sync(0xffffffffu, send, 16);
                    x[i] = ((mask >> i) & 1u) ? mine + other : -INFINITY;   // unscaled logit
                }
            }
            // the row maximum by a tree (not a chain), then in base-2 units (scale > 0)
            float mt[kAtRpl];
#pragma unroll
            for (int i = 0; i < kAtRpl; ++i) mt[i] = x[i];
#pragma unroll
            for (int n = kAtRpl; n > 1; n = (n + 1) / 2)
#pragma unroll
                for (int i = 0; i < n / 2; ++i) mt[i] = fmaxf(mt[i], mt[(n + 1) / 2 + i]);
            float mx = fmaxf(mt[0], __shfl_xor_sync(0xffffffffu, mt[0], 16)) * a.scale_log2;
            float alpha = 1.f;
            if (mx > m_run + kAtTau) {
                alpha = m_run == -INFINITY ? 1.f : exp2f(m_run - mx);
                m_run = mx;
            }
            l_run *= alpha;
            // ---- the rescale factors of all heads, for every warp's quarter of O^T ----
            const int vb = u & 1;
            if (part == 0) alphas[vb * 64 + h] = alpha;
            const bool moved = __any_sync(0xffffffffu, alpha != 1.f);
            if (lane == 0) flags[vb * 4 + q] = moved ? 1 : 0;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(vote_bar);
            if (!ptx::mbar_wait(vote_bar, u & 1)) {
                ok = false;
                break;
            }
            const bool any = (flags[vb * 4] | flags[vb * 4 + 1] | flags[vb * 4 + 2] | flags[vb * 4 + 3]) != 0;
            if (any && u > 0) {
                // O^T holds heads in columns: rescale once PV(u-1) has completed
                if (!ptx::mbar_wait(&pv_done[(u - 1) & 1], ((u - 1) >> 1) & 1)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
#pragma unroll 1
                for (int j = 0; j < CC; ++j) {
                    uint32_t ov[64];
                    const uint32_t addr = lane_base + Cfg::TMEM_O + j * 64;
                    ptx::tmem_ld64(addr, ov);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int hh = 0; hh < 64; ++hh) ov[hh] = __float_as_uint(__uint_as_float(ov[hh]) * alphas[vb * 64 + hh]);
                    ptx::tmem_st32(addr, ov);
                    ptx::tmem_st32(addr + 32, ov + 32);
                }
                ptx::tmem_st_wait();
            }
            // ---- P(u) into buffer u & 1 once PV(u-2), its last reader, has completed ----
            if (u >= 2 && !ptx::mbar_wait(&pv_done[u & 1], ((u - 2) >> 1) & 1)) {
                ok = false;
                break;
            }
            const float ms = m_run == -INFINITY ? 0.f : m_run;
            // P in fp16, two values per conversion; the row sum adds the same rounded values
            uint32_t pw[kAtRpl / 2];
#pragma unroll
            for (int i = 0; i < kAtRpl; i += 2) {
                pw[i / 2] = pack_f16x2(ex2_approx(fmaf(x[i], a.scale_log2, -ms)),
                                       ex2_approx(fmaf(x[i + 1], a.scale_log2, -ms)));
                const float2 pf = __half22float2(*reinterpret_cast<const __half2 *>(&pw[i / 2]));
                l_run += pf.x + pf.y;
            }
            uint8_t *pb = p_buf + (u & 1) * kAtPBytes;
#pragma unroll
            for (int k = 0; k < kAtRpl / 8; ++k)
                *reinterpret_cast<uint4 *>(pb + ptx::sw128_offset(h, (kAtRpl / 8) * part + k)) =
                    make_uint4(pw[4 * k], pw[4 * k + 1], pw[4 * k + 2], pw[4 * k + 3]);
            ptx::fence_proxy_async();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&p_full[u & 1]);
        }
        if (!ok) *abort_flag = 1;
        // ---- the split's results: running max, row sum, unnormalised O ----
        if (ok && !*abort_flag && ptx::mbar_wait(&pv_done[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1)) {
            ptx::tc_fence_after();
            const float l_tot = l_run + __shfl_xor_sync(0xffffffffu, l_run, 16);
            if (part == 0 && h < a.H) {
                a.part_m[pidx0 + h] = m_run;
                a.part_l[pidx0 + h] = l_tot;
            }
#pragma unroll 1
            for (int j = 0; j < CC; ++j) {
                uint32_t ov[64];
                ptx::tmem_ld64(lane_base + Cfg::TMEM_O + j * 64, ov);
                ptx::tmem_ld_wait();
                float *dst = a.part_o + pidx0 * C + j * 128 + 32 * q + lane;
#pragma unroll
                for (int hh = 0; hh < 64; ++hh)
                    if (hh < a.H) dst[(int64_t)hh * C] = __uint_as_float(ov[hh]);
            }
            ptx::tc_fence_before();
        }
    }
    __syncthreads();
    if (warp == kAtMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

}  // namespace lca

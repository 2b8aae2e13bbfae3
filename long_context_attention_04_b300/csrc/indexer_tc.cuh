// indexer_tc.cuh -- lightning-indexer scores on the tcgen05 tensor cores.
//
// DeepSeek-V4 hybrid attention, CSA step two (gxgjx.lffhtl.com/lxrt/355279.html, section
// 混肃穆力机制: a light indexer scores each query against every compressed KV block); [P4]
// zhinnengdao.top section 3.1: 64 indexer query heads of dim 128.  Score (the DeepSeek-V3.2
// lightning-indexer form):  s_j = sum_h w_h * ReLU(q_h . k_j)  for j < floor((pos+1)/m),
// -inf for the entries the query cannot see yet.
//
// The contraction runs transposed, S^T[entry, (query, head)] = K[entry, d] . Q[(query, head), d]^T,
// so that one TMEM lane holds one entry with all its heads: the head reduction
// sum_h w_h ReLU(.) is then a per-thread loop in the epilogue, with no cross-lane traffic.
//   MMA tile: M = 128 entries (A = key tile, K-major, TMA-loaded with 128-byte swizzle),
//             N = QPT queries x H_I heads (B = query tile, K-major, loaded once per group),
//             K = d_I.
// Persistent, warp-specialised, one CTA per SM:
//   warp 0     TMA producer: query tile per (sequence, query group) (two buffers when the key
//              ring keeps 6 stages beside them), key tiles into a ring
//   warp 1     TMEM allocator and MMA issuer (one thread), 2-4 accumulator buffers
//   warps 2..  epilogue: TMEM -> registers, weighted ReLU sum per query, fp32 score store.
//              The 8 epilogue warps form two sets of 4 (a warp group each), set s reading the
//              accumulator buffers b with b mod 2 = s (every other computed tile): one set's
//              TMEM reads overlap the other set's arithmetic, each set has two MMA periods per
//              tile, and 10 warps leave 168 registers a thread.  A set's warp group owns all
//              N columns (whole queries).
// With FUSE (prefill: 4 queries per tile) the epilogue selects each query's top k as the
// scores stream (topk_stream.cuh) instead of storing them: every CTA takes whole query
// groups, so a query's whole row passes through one selection group (the two warp groups,
// one per set, that score its columns).
// Every wait is bounded; a wait that runs out raises LCA_DEVERR_TIMEOUT and the CTA unwinds.
#pragma once

#include "ptx.cuh"
#include "topk_stream.cuh"

namespace lca {

struct IndexerTcArgs {
    int n_q;                    // queries per sequence
    int ratio;                  // m
    int64_t cache_rows;         // entries per sequence in the key cache
    int groups;                 // query groups per sequence: ceil(n_q / QPT)
    int tiles;                  // 128-entry tiles per sequence: ceil(cache_rows / 128)
    int64_t items;              // B * groups * tiles
    const float *w;             // [B][n_q][H_I]
    const int32_t *q_pos;       // [B][n_q]
    float *scores;              // [B][n_q][stride]
    int64_t stride;
    // fused selection (FUSE): k per query, the ascending lists, the candidate buffers
    int k;
    int32_t *out_idx;           // [B][n_q][k]
    uint2 *cand;                // fused selection's candidate buffers (key, index)
    // e4m3 rows (FP8): per (query, head) query scales, per entry key scales
    const float *q_scale;       // [B][n_q][HI]
    const float *k_scale;       // [B] rows of ks_bs
    int64_t ks_bs;
};

template <int DI, int HI, int QPT, bool FUSE = false, bool FP8 = false>
struct IndexerTcConfig {
    static constexpr int N = HI * QPT;                       // MMA N: columns per tile
    static constexpr int ESZ = FP8 ? 1 : 2;                  // bytes per element (e4m3 or bf16)
    static constexpr int BOX = DI * ESZ < 128 ? DI : 128 / ESZ;   // elements per TMA box row
    static constexpr int NBOX = DI / BOX;                    // boxes per row
    static constexpr int ROWB = BOX * ESZ;                   // bytes per box row (128 or 64)
    static constexpr uint32_t SWZ = ROWB == 128 ? ptx::kSwizzle128 : ptx::kSwizzle64;
    static constexpr int KMMA = 32 / ESZ;                    // K per MMA: 32 bytes of a row
    static constexpr int KSTEPS_PER_BOX = BOX / KMMA;
    static constexpr int KSTEPS = DI / KMMA;
    static constexpr int TILE_BYTES = 128 * DI * ESZ;        // one key tile
    static constexpr int SC_BYTES = FP8 ? 128 * 4 : 0;       // its 128 key scales (e4m3)
    static constexpr int Q_BYTES = N * DI * ESZ;             // one query tile
    // epilogue warps: two sets of 4 (a warp group each); set s reads the accumulator buffers
    // b with b mod 2 = s, i.e. every other computed tile
    static constexpr int EPI_WARPS = 8;
    static constexpr int SETS = 2;
    static constexpr int WG_PER_SET = EPI_WARPS / 4 / SETS;  // warp groups per set
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int COLS_PER_WG = N / WG_PER_SET;       // columns one epilogue warp group owns
    static constexpr int QW = COLS_PER_WG / HI;              // queries one warp group scores
    // accumulator buffers in TMEM: the MMA runs up to ACC_BUFS tiles ahead of the epilogue
    static constexpr int ACC_BUFS = 4 * N <= 512 ? 4 : 2;
    static constexpr int TMEM_COLS = ACC_BUFS * N <= 32 ? 32 : ACC_BUFS * N <= 64 ? 64 : ACC_BUFS * N <= 128 ? 128
                                   : ACC_BUFS * N <= 256 ? 256 : 512;
    // fused selection: one selection group per warp group of a set (the same columns in both
    // sets), two candidate buffers per query
    static constexpr int ST_BYTES = FUSE ? (int)((WG_PER_SET * sizeof(StreamWg) + 1023) / 1024 * 1024) : 0;
    static constexpr int64_t CAND_PER_CTA = FUSE ? (int64_t)WG_PER_SET * QW * 2 * kStCap : 0;
    // head weights of the current query group, one copy per epilogue warp (read as broadcasts)
    static constexpr int W_BYTES = EPI_WARPS * COLS_PER_WG * 4;
    static constexpr int SMEM_LIMIT = 227 * 1024 - ST_BYTES - W_BYTES;
    // two query tiles where the key ring still keeps 6 stages (decode: the next sequence's query
    // loads while the MMAs finish the current one, so the ring does not drain at the switch)
    static constexpr int STAGES_2Q = (SMEM_LIMIT - 2 * Q_BYTES - 2048) / (TILE_BYTES + SC_BYTES);
    static constexpr int QBUF = STAGES_2Q >= 6 ? 2 : 1;
    static constexpr int FIXED = QBUF * Q_BYTES + 1024;      // query tiles + barriers
    static constexpr int STAGES_FIT = (SMEM_LIMIT - FIXED - 1024) / (TILE_BYTES + SC_BYTES);
    // key tiles in flight: the stream is latency-bound per SM, so the (half-size) e4m3 tiles
    // get more stages
    static constexpr int STAGES_MAX = FP8 ? 12 : 8;
    static constexpr int STAGES = STAGES_FIT > STAGES_MAX ? STAGES_MAX : STAGES_FIT;
    static constexpr int SMEM_BYTES =
        1024 + QBUF * Q_BYTES + STAGES * (TILE_BYTES + SC_BYTES) + 1024 + ST_BYTES + W_BYTES;
    // a key stage is free once its MMAs are done and, with e4m3 keys, once the epilogue warps
    // that score the tile have read its scales
    static constexpr int EMPTY_COUNT = 1 + (FP8 ? EPI_WARPS / SETS : 0);
    static_assert(N >= 16 && N <= 256 && N % 16 == 0, "MMA N");
    static_assert(!FUSE || (QW <= kStQueries && 4 * SETS == kStWarps), "fused selection group");
    static_assert(ACC_BUFS % SETS == 0, "the sets split the accumulator buffers");
    static_assert(COLS_PER_WG % HI == 0, "a warp group owns whole queries");
    static_assert(HI % 4 == 0, "four partial sums per query");
    static_assert(STAGES >= 2, "ring");
    static_assert(ACC_BUFS * N <= 512, "TMEM");
};

// Position of a work item (sequence b, query group g, tile t) while a CTA walks its contiguous
// range, advanced by increments (no 64-bit division per tile in the loops).
struct ItemCursor {
    int t, g, b;
    int64_t bg;                  // b * groups + g
    int tiles, groups;
    __device__ __forceinline__ ItemCursor(int64_t it, int tiles_, int groups_) : tiles(tiles_), groups(groups_) {
        t = (int)(it % tiles);
        bg = it / tiles;
        b = (int)(bg / groups);
        g = (int)(bg % groups);
    }
    __device__ __forceinline__ void next() {
        if (++t == tiles) {
            t = 0;
            ++bg;
            if (++g == groups) {
                g = 0;
                ++b;
            }
        }
    }
};

template <int DI, int HI, int QPT, bool FUSE = false, bool FP8 = false>
__global__ void __launch_bounds__(IndexerTcConfig<DI, HI, QPT, FUSE, FP8>::THREADS, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                      const __grid_constant__ CUtensorMap smap, IndexerTcArgs a) {
    using Cfg = IndexerTcConfig<DI, HI, QPT, FUSE, FP8>;
    constexpr int N = Cfg::N, STAGES = Cfg::STAGES;
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_tile = base;
    uint8_t *k_ring = base + Cfg::QBUF * Cfg::Q_BYTES;
    float *s_ring = reinterpret_cast<float *>(k_ring + STAGES * Cfg::TILE_BYTES);   // e4m3 key scales
    uint8_t *misc = k_ring + STAGES * (Cfg::TILE_BYTES + Cfg::SC_BYTES);
    uint64_t *full = reinterpret_cast<uint64_t *>(misc);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *acc_empty = acc_full + Cfg::ACC_BUFS;
    uint64_t *q_full = acc_empty + Cfg::ACC_BUFS;
    uint64_t *q_empty = q_full + Cfg::QBUF;
    uint64_t *teardown = q_empty + Cfg::QBUF;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(teardown + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    StreamWg *st = reinterpret_cast<StreamWg *>(misc + 1024);   // FUSE: one per epilogue warp group
    float *w_sm = reinterpret_cast<float *>(misc + 1024 + Cfg::ST_BYTES);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    int64_t it0, it1;
    if constexpr (FUSE) {
        // whole query groups per CTA: a query's row never spans two CTAs
        const int64_t G = a.items / a.tiles;
        it0 = (G * blockIdx.x / gridDim.x) * a.tiles;
        it1 = (G * (blockIdx.x + 1) / gridDim.x) * a.tiles;
    } else {
        const int64_t per = a.items / gridDim.x, rem = a.items % gridDim.x;
        it0 = blockIdx.x * per + (blockIdx.x < rem ? blockIdx.x : rem);
        it1 = it0 + per + (blockIdx.x < rem ? 1 : 0);
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], Cfg::EMPTY_COUNT);
        }
        for (int s = 0; s < Cfg::ACC_BUFS; ++s) {
            ptx::mbar_init(&acc_full[s], 1);
            ptx::mbar_init(&acc_empty[s], Cfg::EPI_WARPS / Cfg::SETS);
        }
        for (int s = 0; s < Cfg::QBUF; ++s) {
            ptx::mbar_init(&q_full[s], 1);
            ptx::mbar_init(&q_empty[s], 1);
        }
        ptx::mbar_init(teardown, 1);
        *abort_flag = 0;
        if constexpr (FUSE) {
            for (int w = 0; w < Cfg::WG_PER_SET; ++w) {
                for (int q = 0; q < kStQueries; ++q) {
                    st[w].kept[q] = 0;
                    for (int v = 0; v < kStWarps; ++v) st[w].wcnt[q][v] = 0;
                    st[w].active[q] = 0;
                    st[w].theta[q] = 0;
                }
                ptx::mbar_init(&st[w].bar, kStWarps);
            }
        }
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();   // the set-up above touches no global memory; everything below may

    // Visible entries of the query group (max over its real queries), same in every role.
    auto group_visible = [&](int b, int g) -> int64_t {
        int64_t v = 0;
        for (int q = 0; q < QPT; ++q) {
            const int qi = g * QPT + q;
            if (qi >= a.n_q) break;
            const int64_t pos = a.q_pos[(int64_t)b * a.n_q + qi];
            int64_t n = pos < 0 ? 0 : (pos + 1) / a.ratio;
            v = n > v ? n : v;
        }
        return v < a.cache_rows ? v : a.cache_rows;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer ----
        if (lane == 0) {
            ptx::tma_prefetch(&kmap);
            ptx::tma_prefetch(&qmap);
            int64_t cur = -1;
            int64_t vis = 0;
            uint32_t fill = 0, groups_loaded = 0;
            ItemCursor ic(it0, a.tiles, a.groups);
            for (int64_t it = it0; it < it1 && !*abort_flag; ++it, ic.next()) {
                const int t = ic.t;
                const int64_t bg = ic.bg;
                const int b = ic.b, g = ic.g;
                if (bg != cur) {
                    const int qb = (int)(groups_loaded % Cfg::QBUF);
                    if (groups_loaded >= (uint32_t)Cfg::QBUF &&
                        !ptx::mbar_wait(&q_empty[qb], ((groups_loaded / Cfg::QBUF) - 1) & 1)) {
                        *abort_flag = 1;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&q_full[qb], Cfg::Q_BYTES);
                    const int qrow = (int)(((int64_t)b * a.n_q + (int64_t)g * QPT) * HI);
#pragma unroll
                    for (int bx = 0; bx < Cfg::NBOX; ++bx)
                        ptx::tma_load_2d(ptx::smem_u32(q_tile + qb * Cfg::Q_BYTES + bx * N * Cfg::ROWB), &qmap,
                                         bx * Cfg::BOX, qrow, &q_full[qb]);
                    ++groups_loaded;
                    cur = bg;
                    vis = group_visible(b, g);
                }
                if ((int64_t)t * 128 >= vis) continue;
                const int s = fill % STAGES;
                if (fill >= (uint32_t)STAGES && !ptx::mbar_wait(&empty[s], ((fill / STAGES) - 1) & 1)) {
                    *abort_flag = 1;
                    break;
                }
                ptx::mbar_arrive_expect_tx(&full[s], Cfg::TILE_BYTES + Cfg::SC_BYTES);
                uint8_t *dst = k_ring + s * Cfg::TILE_BYTES;
                if constexpr (FP8)   // the tile's key scales (rows past the cache are zero-filled)
                    ptx::tma_load_2d(ptx::smem_u32(s_ring + s * 128), &smap, t * 128, b, &full[s]);
#pragma unroll
                for (int bx = 0; bx < Cfg::NBOX; ++bx)
                    ptx::tma_load_3d(ptx::smem_u32(dst + bx * 128 * Cfg::ROWB), &kmap, bx * Cfg::BOX, t * 128, b,
                                     &full[s]);
                ++fill;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issue ----
        if (lane == 0) {
            constexpr uint32_t idesc = FP8 ? ptx::idesc_e4m3(128, N) : ptx::idesc_bf16(128, N, false, false);
            int64_t cur = -1;
            int64_t vis = 0;
            uint32_t use = 0, groups_seen = 0, acc_use[Cfg::ACC_BUFS] = {};
            int acc = 0;
            bool issued = false;
            // descriptors of the ring's and the query tiles' starts; an operand's descriptor is
            // its base plus (byte offset >> 4) in the start-address field (no carry: < 256 KB)
            const uint64_t k_desc = ptx::smem_desc(ptx::smem_u32(k_ring), 16, 8 * Cfg::ROWB, Cfg::SWZ);
            uint64_t q_desc = ptx::smem_desc(ptx::smem_u32(q_tile), 16, 8 * Cfg::ROWB, Cfg::SWZ);
            ItemCursor ic(it0, a.tiles, a.groups);
            for (int64_t it = it0; it < it1 && !*abort_flag; ++it, ic.next()) {
                const int t = ic.t;
                const int64_t bg = ic.bg;
                if (bg != cur) {
                    // the previous query tile is free once the MMAs issued so far finish
                    if (groups_seen > 0) ptx::mma_commit(&q_empty[(groups_seen - 1) % Cfg::QBUF]);
                    const int qb = (int)(groups_seen % Cfg::QBUF);
                    if (!ptx::mbar_wait(&q_full[qb], (groups_seen / Cfg::QBUF) & 1)) {
                        *abort_flag = 1;
                        break;
                    }
                    q_desc = ptx::smem_desc(ptx::smem_u32(q_tile + qb * Cfg::Q_BYTES), 16, 8 * Cfg::ROWB, Cfg::SWZ);
                    ++groups_seen;
                    cur = bg;
                    vis = group_visible(ic.b, ic.g);
                }
                if ((int64_t)t * 128 >= vis) continue;
                if (acc_use[acc] > 0 && !ptx::mbar_wait(&acc_empty[acc], (acc_use[acc] - 1) & 1)) {
                    *abort_flag = 1;
                    break;
                }
                const int s = use % STAGES;
                if (!ptx::mbar_wait(&full[s], (use / STAGES) & 1)) {
                    *abort_flag = 1;
                    break;
                }
                ptx::tc_fence_after();
                const uint64_t a_desc = k_desc + (uint64_t)((s * Cfg::TILE_BYTES) >> 4);
                const uint32_t d = tmem + acc * N;
#pragma unroll
                for (int kk = 0; kk < Cfg::KSTEPS; ++kk) {
                    const int bx = kk / Cfg::KSTEPS_PER_BOX, within = kk % Cfg::KSTEPS_PER_BOX;
                    const uint64_t ad = a_desc + (uint64_t)((bx * 128 * Cfg::ROWB + within * 32) >> 4);
                    const uint64_t bd = q_desc + (uint64_t)((bx * N * Cfg::ROWB + within * 32) >> 4);
                    if constexpr (FP8) ptx::mma_e4m3(d, ad, bd, idesc, kk > 0);
                    else ptx::mma_bf16(d, ad, bd, idesc, kk > 0);
                }
                issued = true;
                ptx::mma_commit(&empty[s]);
                ptx::mma_commit(&acc_full[acc]);
                ++acc_use[acc];
                acc = acc + 1 == Cfg::ACC_BUFS ? 0 : acc + 1;
                ++use;
            }
            if (issued) {
                // drain: every MMA this thread issued completes before TMEM is released
                ptx::mma_commit(teardown);
                ptx::mbar_wait(teardown, 0);
            }
        }
    } else {
        // -------------------------------------------------------------- epilogue ----
        const int ew = warp - 2;                         // 0 .. EPI_WARPS-1
        const int set = ew / (4 * Cfg::WG_PER_SET);      // the accumulator buffer this warp reads
        const int wg = (ew >> 2) % Cfg::WG_PER_SET;      // its warp group within the set
        const int quarter = warp & 3;                    // TMEM lane quarter this warp may access
        const int col0 = wg * Cfg::COLS_PER_WG;          // first column of this warp group
        constexpr int QW = Cfg::QW;                      // queries this warp group scores
        const int row = quarter * 32 + lane;             // tile row == TMEM lane
        int64_t cur = -1;
        int64_t vis = 0;
        int nv[QW];                                      // visible entries of each query
        float *wr = w_sm + ew * Cfg::COLS_PER_WG;        // head weights of this warp group's queries
        uint32_t acc_use[Cfg::ACC_BUFS] = {};
        int acc = 0;
        // fused selection: the selection group's state (one per warp group of a set), this warp's
        // segment and thread index in it, the candidate buffers, and this warp's copies of its
        // segment counts, thresholds and active buffers
        const int wseg = set * 4 + (ew & 3);
        const int wtid = wseg * 32 + lane;
        uint2 *cand = FUSE ? a.cand + ((int64_t)blockIdx.x * Cfg::WG_PER_SET + wg) * (QW * 2 * kStCap) : nullptr;
        uint32_t st_phase = 0;
        // (the thresholds and active buffers are read from the group's shared state: they change
        // only at checkpoints, and registers are scarce)
        int my_cnt[QW];
#pragma unroll
        for (int q = 0; q < QW; ++q) my_cnt[q] = 0;
        constexpr int CH = Cfg::COLS_PER_WG < 32 ? Cfg::COLS_PER_WG : 32;   // TMEM columns per load
        constexpr int NCH = Cfg::COLS_PER_WG / CH;
        auto tmem_ld_chunk = [&](uint32_t addr, uint32_t *r) {
            if constexpr (CH == 32) ptx::tmem_ld32(addr, r);
            else if constexpr (CH == 16) ptx::tmem_ld16(addr, r);
            else ptx::tmem_ld8(addr, r);
        };
        uint32_t fidx = 0;                               // computed tiles so far (= key fills)
        ItemCursor ic(it0, a.tiles, a.groups);
        for (int64_t it = it0; it < it1 && !*abort_flag; ++it, ic.next()) {
            const int t = ic.t;
            const int64_t bg = ic.bg;
            const int b = ic.b, g = ic.g;
            if (bg != cur) {
                cur = bg;
                vis = group_visible(b, g);
                __syncwarp();                            // the last group's weights are read
                for (int c = lane; c < Cfg::COLS_PER_WG; c += 32) {
                    const int qi = g * QPT + col0 / HI + c / HI;
                    const int64_t wi = ((int64_t)b * a.n_q + qi) * HI + c % HI;
                    // e4m3 queries: the (non-negative) query scale moves out of the ReLU into the weight
                    wr[c] = qi < a.n_q ? (FP8 ? __ldg(a.w + wi) * __ldg(a.q_scale + wi) : __ldg(a.w + wi)) : 0.f;
                }
                __syncwarp();
#pragma unroll
                for (int q = 0; q < QW; ++q) {
                    const int qi = g * QPT + col0 / HI + q;
                    int64_t n = 0;
                    if (qi < a.n_q) {
                        const int64_t pos = a.q_pos[(int64_t)b * a.n_q + qi];
                        n = pos < 0 ? 0 : (pos + 1) / a.ratio;
                        if (n > a.cache_rows) {
                            if (threadIdx.x == 64 && t == 0) raise_error(LCA_DEVERR_VISIBLE_RANGE);
                            n = a.cache_rows;
                        }
                    }
                    nv[q] = (int)n;
                }
            }
            const int64_t j = (int64_t)t * 128 + row;
            float sc[QW];
#pragma unroll
            for (int q = 0; q < QW; ++q) sc[q] = 0.f;
            const bool computed = (int64_t)t * 128 < vis;
            // this warp's set handles the tile: a computed tile's accumulator buffer, else its parity
            const bool mine = Cfg::SETS == 1 || (computed ? acc % Cfg::SETS == set : t % Cfg::SETS == set);
            if (computed && !mine) {
                ++acc_use[acc];
                acc = acc + 1 == Cfg::ACC_BUFS ? 0 : acc + 1;
                ++fidx;
            } else if (computed) {
                // e4m3 keys: the entry's scale from the tile's key stage (its copy has landed when
                // the stage's full phase completes; the stage is refilled only after this warp's
                // arrival on its empty barrier)
                float ks = 1.f;
                if constexpr (FP8) {
                    const int ss = (int)(fidx % STAGES);
                    if (!ptx::mbar_wait(&full[ss], (fidx / STAGES) & 1)) {
                        *abort_flag = 1;
                        break;
                    }
                    ks = s_ring[ss * 128 + row];
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&empty[ss]);
                }
                ++fidx;
                if (!ptx::mbar_wait(&acc_full[acc], acc_use[acc] & 1)) {
                    *abort_flag = 1;
                    break;
                }
                ptx::tc_fence_after();
                // chunks of CH columns, the next chunk's load in flight while this one is summed;
                // four partial sums per query (head h goes to sum h mod 4), added pairwise at the
                // end, so the FMA chains are a quarter as long
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * N + col0;
                float ps[QW][4];
#pragma unroll
                for (int q = 0; q < QW; ++q)
#pragma unroll
                    for (int v = 0; v < 4; ++v) ps[q][v] = 0.f;
                uint32_t rb[2][CH];
                tmem_ld_chunk(taddr, rb[0]);
                ptx::tmem_ld_wait();
                ptx::reg_fence<CH>(rb[0]);
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    if (c + 1 < NCH) {
                        tmem_ld_chunk(taddr + (c + 1) * CH, rb[(c + 1) & 1]);
                    } else {                             // every TMEM load of this tile has landed
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(&acc_empty[acc]);
                    }
#pragma unroll
                    for (int u = 0; u < CH; u += 4) {
                        const float4 w4 = *reinterpret_cast<const float4 *>(wr + c * CH + u);
                        const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int v = 0; v < 4; ++v)
                            ps[(c * CH + u + v) / HI][v] =
                                fmaf(wv[v], fmaxf(__uint_as_float(rb[c & 1][u + v]), 0.f), ps[(c * CH + u + v) / HI][v]);
                    }
                    if (c + 1 < NCH) {
                        ptx::tmem_ld_wait();
                        ptx::reg_fence<CH>(rb[(c + 1) & 1]);
                    }
                }
#pragma unroll
                for (int q = 0; q < QW; ++q) sc[q] = (ps[q][0] + ps[q][1]) + (ps[q][2] + ps[q][3]);
                if constexpr (FP8) {
                    // e4m3 keys: the entry's (non-negative) scale multiplies the head sum
#pragma unroll
                    for (int q = 0; q < QW; ++q) sc[q] *= ks;
                }
                ++acc_use[acc];
                acc = acc + 1 == Cfg::ACC_BUFS ? 0 : acc + 1;
            }
            if constexpr (FUSE) {
                const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
                for (int q = 0; q < QW; ++q) {
                    // append the scores at or above the query's threshold to this warp's segment
                    const uint32_t key = ordered_key(sc[q]);
                    const bool pass = mine && computed && j < nv[q] && key >= st[wg].theta[q];
                    const uint32_t m = __ballot_sync(0xffffffffu, pass);
                    if (m) {
                        const int pos = my_cnt[q] + __popc(m & lt);
                        if (pass) {
                            if (pos < kStSeg)
                                st_segment(st_buffer(cand, q, st[wg].active[q]), wseg)[pos] =
                                    make_uint2(key, (uint32_t)j);
                            else
                                raise_error(LCA_DEVERR_SELECT);
                        }
                        my_cnt[q] += __popc(m);
                    }
                }
                const bool last = t == a.tiles - 1;
                if (last || (t + 1) % kStSyncTiles == 0) {
                    StreamWg &S = st[wg];
                    if (lane == 0)
#pragma unroll
                        for (int q = 0; q < QW; ++q) S.wcnt[q][wseg] = my_cnt[q];
                    bool fine = wg_sync(S, st_phase);          // every warp's counts are published
                    // a query whose segments could overflow before the next check is compacted;
                    // every warp reads the counts before any warp publishes again (second
                    // barrier), so all of them take the same branches
                    bool full[QW];
#pragma unroll
                    for (int q = 0; q < QW; ++q) {
                        int mx = 0;
#pragma unroll
                        for (int v = 0; v < kStWarps; ++v) mx = max(mx, S.wcnt[q][v]);
                        full[q] = mx > kStSegLimit;
                    }
                    fine = fine && wg_sync(S, st_phase);
                    bool changed = false;
#pragma unroll
                    for (int q = 0; q < QW; ++q)
                        if (full[q] && fine) {
                            fine = wg_compact(S, st_phase, wtid, cand, q, a.k);
                            changed = true;
                        }
                    if (last) {
#pragma unroll
                        for (int q = 0; q < QW; ++q) {
                            const int qi = g * QPT + col0 / HI + q;
                            int32_t *out = qi < a.n_q ? a.out_idx + ((int64_t)b * a.n_q + qi) * a.k : nullptr;
                            if (fine) fine = wg_finish(S, st_phase, wtid, cand, q, a.k, out);
                        }
                        changed = true;
                    }
                    if (!fine) {
                        *abort_flag = 1;
                        break;
                    }
                    if (changed)
#pragma unroll
                        for (int q = 0; q < QW; ++q) {
                            my_cnt[q] = S.wcnt[q][wseg];
                        }
                }
            } else if (mine && j < a.cache_rows) {
#pragma unroll
                for (int q = 0; q < QW; ++q) {
                    const int qi = g * QPT + col0 / HI + q;
                    if (qi < a.n_q)
                        a.scores[((int64_t)b * a.n_q + qi) * a.stride + j] = j < nv[q] ? sc[q] : -INFINITY;
                }
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

}  // namespace lca

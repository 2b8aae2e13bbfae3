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
//   warps 2..  epilogue: TMEM -> registers, weighted ReLU sum per query, fp32 score store
// Every wait is bounded; a wait that runs out raises LCA_DEVERR_TIMEOUT and the CTA unwinds.
#pragma once

#include "ptx.cuh"

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
};

template <int DI, int HI, int QPT>
struct IndexerTcConfig {
    static constexpr int N = HI * QPT;                       // MMA N: columns per tile
    static constexpr int BOX = DI < 64 ? DI : 64;            // elements per TMA box row
    static constexpr int NBOX = DI / BOX;                    // boxes per row
    static constexpr int ROWB = BOX * 2;                     // bytes per box row (128 or 64)
    static constexpr uint32_t SWZ = ROWB == 128 ? ptx::kSwizzle128 : ptx::kSwizzle64;
    static constexpr int KSTEPS_PER_BOX = BOX / 16;
    static constexpr int KSTEPS = DI / 16;
    static constexpr int TILE_BYTES = 128 * DI * 2;          // one key tile
    static constexpr int Q_BYTES = N * DI * 2;               // one query tile
    static constexpr int EPI_WARPS = N > 64 ? 8 : 4;
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int COLS_PER_WG = N / (EPI_WARPS / 4);  // columns one epilogue warp group owns
    // accumulator buffers in TMEM: the MMA runs up to ACC_BUFS tiles ahead of the epilogue
    static constexpr int ACC_BUFS = 4 * N <= 512 ? 4 : 2;
    static constexpr int TMEM_COLS = ACC_BUFS * N <= 32 ? 32 : ACC_BUFS * N <= 64 ? 64 : ACC_BUFS * N <= 128 ? 128
                                   : ACC_BUFS * N <= 256 ? 256 : 512;
    static constexpr int SMEM_LIMIT = 227 * 1024;
    // two query tiles where the key ring still keeps 6 stages (decode: the next sequence's query
    // loads while the MMAs finish the current one, so the ring does not drain at the switch)
    static constexpr int STAGES_2Q = (SMEM_LIMIT - 2 * Q_BYTES - 2048) / TILE_BYTES;
    static constexpr int QBUF = STAGES_2Q >= 6 ? 2 : 1;
    static constexpr int FIXED = QBUF * Q_BYTES + 1024;      // query tiles + barriers
    static constexpr int STAGES_FIT = (SMEM_LIMIT - FIXED - 1024) / TILE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 8 ? 8 : STAGES_FIT;
    static constexpr int SMEM_BYTES = 1024 + QBUF * Q_BYTES + STAGES * TILE_BYTES + 1024;
    static_assert(N >= 16 && N <= 256 && N % 16 == 0, "MMA N");
    static_assert(COLS_PER_WG % HI == 0, "a warp group owns whole queries");
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

template <int DI, int HI, int QPT>
__global__ void __launch_bounds__(IndexerTcConfig<DI, HI, QPT>::THREADS, 1)
    indexer_tc_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                      IndexerTcArgs a) {
    using Cfg = IndexerTcConfig<DI, HI, QPT>;
    constexpr int N = Cfg::N, STAGES = Cfg::STAGES;
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *q_tile = base;
    uint8_t *k_ring = base + Cfg::QBUF * Cfg::Q_BYTES;
    uint8_t *misc = k_ring + STAGES * Cfg::TILE_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(misc);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *acc_empty = acc_full + Cfg::ACC_BUFS;
    uint64_t *q_full = acc_empty + Cfg::ACC_BUFS;
    uint64_t *q_empty = q_full + Cfg::QBUF;
    uint64_t *teardown = q_empty + Cfg::QBUF;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(teardown + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t per = a.items / gridDim.x, rem = a.items % gridDim.x;
    const int64_t it0 = blockIdx.x * per + (blockIdx.x < rem ? blockIdx.x : rem);
    const int64_t it1 = it0 + per + (blockIdx.x < rem ? 1 : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < Cfg::ACC_BUFS; ++s) {
            ptx::mbar_init(&acc_full[s], 1);
            ptx::mbar_init(&acc_empty[s], Cfg::EPI_WARPS);
        }
        for (int s = 0; s < Cfg::QBUF; ++s) {
            ptx::mbar_init(&q_full[s], 1);
            ptx::mbar_init(&q_empty[s], 1);
        }
        ptx::mbar_init(teardown, 1);
        *abort_flag = 0;
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
                ptx::mbar_arrive_expect_tx(&full[s], Cfg::TILE_BYTES);
                uint8_t *dst = k_ring + s * Cfg::TILE_BYTES;
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
            constexpr uint32_t idesc = ptx::idesc_bf16(128, N, false, false);
            int64_t cur = -1;
            int64_t vis = 0;
            uint32_t use = 0, groups_seen = 0, acc_use[Cfg::ACC_BUFS] = {};
            int acc = 0;
            bool issued = false;
            uint32_t q_addr = ptx::smem_u32(q_tile);
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
                    q_addr = ptx::smem_u32(q_tile + qb * Cfg::Q_BYTES);
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
                const uint32_t a_addr = ptx::smem_u32(k_ring + s * Cfg::TILE_BYTES);
                const uint32_t d = tmem + acc * N;
#pragma unroll
                for (int kk = 0; kk < Cfg::KSTEPS; ++kk) {
                    const int bx = kk / Cfg::KSTEPS_PER_BOX, within = kk % Cfg::KSTEPS_PER_BOX;
                    const uint64_t ad = ptx::smem_desc(a_addr + bx * 128 * Cfg::ROWB + within * 32, 16,
                                                       8 * Cfg::ROWB, Cfg::SWZ);
                    const uint64_t bd = ptx::smem_desc(q_addr + bx * N * Cfg::ROWB + within * 32, 16,
                                                       8 * Cfg::ROWB, Cfg::SWZ);
                    ptx::mma_bf16(d, ad, bd, idesc, kk > 0);
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
        const int quarter = warp & 3;                    // TMEM lane quarter this warp may access
        const int col0 = (ew / 4) * Cfg::COLS_PER_WG;    // first column of this warp group
        constexpr int QW = Cfg::COLS_PER_WG / HI;        // queries this warp group scores
        const int row = quarter * 32 + lane;             // tile row == TMEM lane
        int64_t cur = -1;
        int64_t vis = 0;
        int64_t nv[QW];
        float wr[Cfg::COLS_PER_WG];                      // head weights of this group's queries
        uint32_t acc_use[Cfg::ACC_BUFS] = {};
        int acc = 0;
        ItemCursor ic(it0, a.tiles, a.groups);
        for (int64_t it = it0; it < it1 && !*abort_flag; ++it, ic.next()) {
            const int t = ic.t;
            const int64_t bg = ic.bg;
            const int b = ic.b, g = ic.g;
            if (bg != cur) {
                cur = bg;
                vis = group_visible(b, g);
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
                    nv[q] = n;
                    const float *wq = a.w + ((int64_t)b * a.n_q + qi) * HI;
#pragma unroll
                    for (int h = 0; h < HI; ++h) wr[q * HI + h] = qi < a.n_q ? __ldg(wq + h) : 0.f;
                }
            }
            const int64_t j = (int64_t)t * 128 + row;
            float sc[QW];
#pragma unroll
            for (int q = 0; q < QW; ++q) sc[q] = 0.f;
            if ((int64_t)t * 128 < vis) {
                if (!ptx::mbar_wait(&acc_full[acc], acc_use[acc] & 1)) {
                    *abort_flag = 1;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + acc * N + col0;
                // several columns per TMEM round trip (all loads issued before one wait)
                constexpr int CB = Cfg::COLS_PER_WG <= 64 ? Cfg::COLS_PER_WG : 32;
#pragma unroll
                for (int c0 = 0; c0 < Cfg::COLS_PER_WG; c0 += CB) {
                    uint32_t r[CB];
#pragma unroll
                    for (int c = 0; c < CB; c += 16) ptx::tmem_ld16(taddr + c0 + c, r + c);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < CB; ++u)
                        sc[(c0 + u) / HI] = fmaf(wr[c0 + u], fmaxf(__uint_as_float(r[u]), 0.f), sc[(c0 + u) / HI]);
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&acc_empty[acc]);
                ++acc_use[acc];
                acc = acc + 1 == Cfg::ACC_BUFS ? 0 : acc + 1;
            }
            if (j < a.cache_rows) {
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

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
//   S^T[row, head]  = KV[row, c] . Qhat[head, c]^T        (M = 128 rows,  N = 64, K = c)
//   O^T[c, head]   += KV[row, c]^T . P^T[row, head]       (M = 128 c,     N = 64, K = 128 rows)
// The same 128-byte-swizzled shared-memory tile serves as the K-major A operand of the first
// product and the MN-major A operand of the second.  S^T (two buffers) and O^T (c/128
// chunks) live in TMEM; P^T goes through shared memory in bf16.
//
// The normalised, rotated query is split into bf16 hi + lo parts (q = hi + lo to ~16 bits)
// and S^T accumulates KV.hi^T + KV.lo^T in fp32: a single bf16 query would put a relative
// error of 2^-9 on every logit, comparable to the bf16 rounding of the output itself.
// Shared memory holds the 64 KB hi tile and a ring of three 48 KB slots, each a 128-row x
// 128-c KV chunk plus the matching 16 KB lo chunk (copied from this CTA's workspace image).
// A 128-row tile at c = 512 does not fit twice, so each tile is streamed twice, once for S
// and once for PV, the second time from L2.  HBM traffic stays one pass.
//
// Roles (one CTA per (query, split), one CTA per SM):
//   warps 0-3   producers: 16-byte cp.async gathers of rows (compressed entries by index or
//               by position, window rows from the ring) into the swizzled slots
//   warps 4-11  softmax: one TMEM lane (row) per thread, 32 heads per thread; online softmax
//               in base 2 with a conditional rescale (the running max moves only when a
//               logit exceeds it by more than 2^8), P^T rows to shared memory
//   warp 12     TMEM allocator and MMA issuer
// The split's unnormalised O, running max and row sum go to the workspace; combine_kernel
// merges the splits with the sink and applies the output RoPE(-pos).
// Every wait is bounded; a wait that runs out raises LCA_DEVERR_TIMEOUT and the CTA unwinds.
#pragma once

#include "attend_common.cuh"
#include "ptx.cuh"

namespace lca {

constexpr int kAtHP = 64;            // padded heads (MMA N)
constexpr int kAtTile = 128;         // rows per tile (MMA M of S^T)
constexpr int kAtSlots = 3;          // chunk slots in the ring
constexpr int kAtChunkBytes = 128 * 128 * 2;            // KV chunk: 128 rows x 128 c
constexpr int kAtLoChunkBytes = kAtHP * 128 * 2;        // q lo chunk: 64 heads x 128 c
constexpr int kAtSlotBytes = kAtChunkBytes + kAtLoChunkBytes;
constexpr int kAtProducerWarps = 4;
constexpr int kAtSoftmaxWarps = 8;
constexpr int kAtMmaWarp = kAtProducerWarps + kAtSoftmaxWarps;
constexpr int kAtThreads = 32 * (kAtMmaWarp + 1);
constexpr float kAtTau = 8.0f;       // log2 headroom before the running max must move

template <int C>
struct AttendTcConfig {
    static constexpr int CC = C / 128;                        // c chunks per row
    static constexpr int Q_BYTES = kAtHP * C * 2;
    static constexpr int P_BYTES = kAtTile * kAtHP * 2;       // one P^T buffer (16 KB)
    static constexpr int TMEM_S = 0;                          // two S^T buffers: columns 0..127
    static constexpr int TMEM_O = 2 * kAtHP;                  // O^T chunk j at TMEM_O + 64 j
    static constexpr int TMEM_NEED = TMEM_O + CC * kAtHP;
    static constexpr int TMEM_COLS = TMEM_NEED <= 256 ? 256 : 512;
    static constexpr int LO_IMAGE_BYTES = CC * kAtLoChunkBytes;  // per CTA, in the workspace
    static constexpr int MISC = 1280;                          // barriers, votes, cross-warp maxima
    static constexpr int SMEM_BYTES = MISC + 1024 + Q_BYTES + kAtSlots * kAtSlotBytes + P_BYTES;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

// Row code of one row of a query's row list: entry index, 0x80000000 | ring slot for a
// window row, or 0xffffffff for a masked row.
__device__ __forceinline__ uint32_t row_code(const AttendArgs &a, const RowList &L, int64_t R, bool report) {
    if (R >= L.total()) return 0xffffffffu;
    if (R < L.n_comp) {
        const int64_t j = L.idx ? (int64_t)__ldg(L.idx + R) : R;
        if (j < 0) return 0xffffffffu;
        if (j >= a.cache_rows) {
            if (report) raise_error(LCA_DEVERR_INDEX_RANGE);
            return 0xffffffffu;
        }
        return (uint32_t)j;
    }
    const int64_t t = L.win_begin + (R - L.n_comp);
    return 0x80000000u | (uint32_t)(t % a.win_cap);
}

template <int C>
__global__ void __launch_bounds__(kAtThreads, 1) attend_tc_kernel(AttendArgs a) {
    using Cfg = AttendTcConfig<C>;
    constexpr int CC = Cfg::CC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *misc = smem_raw;
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw + Cfg::MISC) + 1023) &
                                                ~uintptr_t(1023));
    uint8_t *q_tile = base;                                   // hi: C/64 boxes of [64 heads x 128 B]
    uint8_t *ring = q_tile + Cfg::Q_BYTES;                    // slots: KV [2 x 128 rows x 128 B] + lo chunk
    uint8_t *p_buf = ring + kAtSlots * kAtSlotBytes;          // [128 rows x 128 B]
    uint64_t *full = reinterpret_cast<uint64_t *>(misc);
    uint64_t *empty = full + kAtSlots;
    uint64_t *s_full = empty + kAtSlots;
    uint64_t *s_empty = s_full + 2;
    uint64_t *p_full = s_empty + 2;
    uint64_t *pv_done = p_full + 2;
    uint64_t *vote_bar = pv_done + 2;
    uint64_t *red_bar = vote_bar + 1;
    uint64_t *teardown = red_bar + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(teardown + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int *votes = reinterpret_cast<int *>(misc + 192);                  // [2][8]
    float *red = reinterpret_cast<float *>(misc + 256);                // [8][32]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int unit = blockIdx.x, split = blockIdx.y;
    const int b = unit / a.n_q, qi = unit % a.n_q;
    const RowList L = make_row_list(a, b, qi);
    int64_t t0, t1;
    split_range(L.total(), kAtTile, split, a.splits, t0, t1);
    const int64_t pidx0 = ((int64_t)unit * a.splits + split) * a.H;
    uint8_t *lo_img = a.q_lo_img + ((int64_t)unit * a.splits + split) * Cfg::LO_IMAGE_BYTES;

    if (t0 >= t1) {   // nothing to do for this split: mark it empty for the combine
        for (int h = threadIdx.x; h < a.H; h += blockDim.x) {
            a.part_m[pidx0 + h] = -INFINITY;
            a.part_l[pidx0 + h] = 0.f;
        }
        return;
    }

    // ---- set-up: barriers, TMEM, the normalised and rotated query tile ----
    if (threadIdx.x == 0) {
        for (int s = 0; s < kAtSlots; ++s) {
            ptx::mbar_init(&full[s], 32 * kAtProducerWarps);
            ptx::mbar_init(&empty[s], 1);
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
    for (int h = warp; h < kAtHP; h += kAtThreads / 32) {
        constexpr int EPL = C / 32;
        float v[EPL];
        if (h < a.H) {
            q_hat_warp<C>(a, a.q + ((int64_t)unit * a.H + h) * C, L.pos, v);
        } else {
#pragma unroll
            for (int u = 0; u < EPL; ++u) v[u] = 0.f;
        }
        // hi = bf16(q), lo = bf16(q - hi); lane holds elements [lane*EPL, lane*EPL + EPL)
        float lo[EPL];
#pragma unroll
        for (int u = 0; u < EPL; ++u) {
            const float hi = __bfloat162float(__float2bfloat16_rn(v[u]));
            lo[u] = v[u] - hi;
            v[u] = hi;
        }
        // hi -> resident tile (box e/64); lo -> image: chunk e/128, box (e%128)/64
        if constexpr (EPL >= 8) {
#pragma unroll
            for (int u = 0; u < EPL; u += 8) {
                const int e = lane * EPL + u;
                const uint32_t off = ptx::sw128_offset(h, (e % 64) / 8);
                *reinterpret_cast<uint4 *>(q_tile + (e / 64) * (kAtHP * 128) + off) = pack8(v + u);
                *reinterpret_cast<uint4 *>(lo_img + (e / 64) * (kAtHP * 128) + off) = pack8(lo + u);
            }
        } else {
            const int e = lane * EPL;   // 4 elements: half a chunk
            const uint32_t off = ptx::sw128_offset(h, (e % 64) / 8) + (e % 8) * 2;
            *reinterpret_cast<uint2 *>(q_tile + (e / 64) * (kAtHP * 128) + off) =
                make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
            *reinterpret_cast<uint2 *>(lo_img + (e / 64) * (kAtHP * 128) + off) =
                make_uint2(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]));
        }
    }
    ptx::fence_proxy_async();
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int n_tiles = (int)(t1 - t0);

    if (warp < kAtProducerWarps) {
        // ------------------------------------------------------------ producers ----
        const __nv_bfloat16 *kv_b = L.kv, *win_b = L.win;
        const int sub_row = warp * 2 + (lane >> 4);   // row within an 8-row stripe
        const int piece = lane & 15;                  // 16-byte piece of the 256-byte chunk row
        uint32_t cur[16], nxt[16];
        uint32_t issued = 0;                          // chunk loads issued
        uint32_t arrived = 0;                         // chunk loads signalled complete
        auto load_chunk = [&](const uint32_t *codes, int j, bool with_lo) -> bool {
            const int s = issued % kAtSlots;
            if (issued >= (uint32_t)kAtSlots && !ptx::mbar_wait(&empty[s], ((issued / kAtSlots) - 1) & 1))
                return false;
            uint8_t *slot = ring + s * kAtSlotBytes;
            if (with_lo) {   // the lo part of query chunk j (16 KB, already swizzled)
                const uint32_t lo_dst = ptx::smem_u32(slot + kAtChunkBytes);
                const uint8_t *lo_src = lo_img + j * kAtLoChunkBytes;
#pragma unroll
                for (int i = 0; i < kAtLoChunkBytes / 16 / (32 * kAtProducerWarps); ++i) {
                    const int piece16 = i * (32 * kAtProducerWarps) + threadIdx.x;
                    ptx::cp_async16(lo_dst + piece16 * 16, lo_src + piece16 * 16, 16);
                }
            }
            const uint32_t dst0 = ptx::smem_u32(slot) + (piece >> 3) * (128 * 128);
#pragma unroll
            for (int it = 0; it < 16; ++it) {
                const int r = it * 8 + sub_row;
                const uint32_t code = codes[it];
                const __nv_bfloat16 *src = kv_b;
                uint32_t bytes = 0;
                if (code != 0xffffffffu) {
                    src = (code & 0x80000000u) ? win_b + (int64_t)(code & 0x7fffffffu) * C
                                               : kv_b + (int64_t)code * C;
                    src += j * 128 + piece * 8;
                    bytes = 16;
                }
                ptx::cp_async16(dst0 + ptx::sw128_offset(r, piece & 7), src, bytes);
            }
            ptx::cp_async_commit();
            ++issued;
            // signal the chunk issued two loads ago (its copies are complete now)
            if (issued >= 3) {
                ptx::cp_async_wait<2>();
                ptx::fence_proxy_async();
                ptx::mbar_arrive(&full[arrived % kAtSlots]);
                ++arrived;
            }
            return true;
        };
        auto codes_of = [&](uint32_t *codes, int64_t t) {
#pragma unroll
            for (int it = 0; it < 16; ++it) codes[it] = row_code(a, L, t * kAtTile + it * 8 + sub_row, piece == 0);
        };
        bool ok = true;
        codes_of(cur, t0);
        for (int j = 0; j < CC && ok; ++j) ok = load_chunk(cur, j, true);
        for (int64_t t = t0 + 1; t < t1 && ok && !*abort_flag; ++t) {
            codes_of(nxt, t);
            for (int j = 0; j < CC && ok; ++j) ok = load_chunk(nxt, j, true);      // S(t)
            for (int j = 0; j < CC && ok; ++j) ok = load_chunk(cur, j, false);     // PV(t-1)
#pragma unroll
            for (int it = 0; it < 16; ++it) cur[it] = nxt[it];
        }
        for (int j = 0; j < CC && ok; ++j) ok = load_chunk(cur, j, false);         // PV(t1-1)
        if (!ok) *abort_flag = 1;
        ptx::cp_async_wait_all();
        ptx::fence_proxy_async();
        while (arrived < issued) {
            ptx::mbar_arrive(&full[arrived % kAtSlots]);
            ++arrived;
        }
    } else if (warp == kAtMmaWarp) {
        // ------------------------------------------------------------- MMA issue ----
        if (lane == 0) {
            constexpr uint32_t idesc_s = ptx::idesc_bf16(128, kAtHP, false, false);
            constexpr uint32_t idesc_o = ptx::idesc_bf16(128, kAtHP, true, true);
            const uint32_t q_addr = ptx::smem_u32(q_tile);
            uint32_t used = 0;   // chunk slots consumed
            bool ok = true;
            auto take = [&]() -> uint32_t {   // wait for the next chunk; returns its smem address
                const int s = used % kAtSlots;
                if (!ptx::mbar_wait(&full[s], (used / kAtSlots) & 1)) return 0;
                ptx::tc_fence_after();
                return ptx::smem_u32(ring + s * kAtSlotBytes);
            };
            auto issue_s = [&](int u) -> bool {   // S^T of relative tile u
                const int buf = u & 1;
                if (u >= 2 && !ptx::mbar_wait(&s_empty[buf], ((u >> 1) - 1) & 1)) return false;
                ptx::tc_fence_after();
                for (int j = 0; j < CC; ++j) {
                    const uint32_t slot = take();
                    if (!slot) return false;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = ptx::smem_desc(slot + (kk >> 2) * (128 * 128) + (kk & 3) * 32, 16, 1024,
                                                           ptx::kSwizzle128);
                        const uint64_t bh = ptx::smem_desc(q_addr + (2 * j + (kk >> 2)) * (kAtHP * 128) +
                                                               (kk & 3) * 32,
                                                           16, 1024, ptx::kSwizzle128);
                        const uint64_t bl = ptx::smem_desc(slot + kAtChunkBytes + (kk >> 2) * (kAtHP * 128) +
                                                               (kk & 3) * 32,
                                                           16, 1024, ptx::kSwizzle128);
                        const uint32_t d = tmem + Cfg::TMEM_S + buf * kAtHP;
                        ptx::mma_bf16(d, ad, bh, idesc_s, (j > 0 || kk > 0));
                        ptx::mma_bf16(d, ad, bl, idesc_s, 1);
                    }
                    ptx::mma_commit(&empty[used % kAtSlots]);
                    ++used;
                }
                ptx::mma_commit(&s_full[buf]);
                return true;
            };
            auto issue_pv = [&](int u) -> bool {   // O^T += V^T P^T of relative tile u
                const int buf = u & 1;
                if (!ptx::mbar_wait(&p_full[buf], (u >> 1) & 1)) return false;
                ptx::tc_fence_after();
                const uint32_t p_addr = ptx::smem_u32(p_buf);
                for (int j = 0; j < CC; ++j) {
                    const uint32_t slot = take();
                    if (!slot) return false;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint64_t ad = ptx::smem_desc(slot + kk * 2048, 128 * 128, 1024, ptx::kSwizzle128);
                        const uint64_t bd = ptx::smem_desc(p_addr + kk * 2048, 128 * 128, 1024, ptx::kSwizzle128);
                        ptx::mma_bf16(tmem + Cfg::TMEM_O + j * kAtHP, ad, bd, idesc_o, (u > 0 || kk > 0));
                    }
                    ptx::mma_commit(&empty[used % kAtSlots]);
                    ++used;
                }
                ptx::mma_commit(&pv_done[buf]);
                return true;
            };
            ok = issue_s(0);
            for (int u = 1; u < n_tiles && ok && !*abort_flag; ++u) {
                ok = issue_s(u);
                if (ok) ok = issue_pv(u - 1);
            }
            if (ok && !*abort_flag) ok = issue_pv(n_tiles - 1);
            if (!ok) *abort_flag = 1;
            ptx::mma_commit(teardown);
            ptx::mbar_wait(teardown, 0);
        }
    } else {
        // -------------------------------------------------------------- softmax ----
        const int sw = warp - kAtProducerWarps;      // 0..7
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
        for (int u = 0; u < n_tiles && !*abort_flag; ++u) {
            const int buf = u & 1;
            if (!ptx::mbar_wait(&s_full[buf], (u >> 1) & 1)) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            float x[32];
            {
                uint32_t v[32];
                ptx::tmem_ld32(lane_addr + Cfg::TMEM_S + buf * kAtHP + half * 32, v);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 32; ++h) x[h] = __uint_as_float(v[h]);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&s_empty[buf]);
            const bool valid = row_code(a, L, (t0 + u) * kAtTile + r, false) != 0xffffffffu;
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
                // O^T holds data once PV of the previous tile is done: wait for it, then rescale
                if (u > 0) {
                    if (!ptx::mbar_wait(&pv_done[(u - 1) & 1], ((u - 1) >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                }
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
            // probabilities of this row, written as a bf16 P^T row (32 heads = 4 chunks) into the
            // single P buffer once PV of the previous tile has read it
            if (u >= 1) {
                if (!ptx::mbar_wait(&pv_done[(u - 1) & 1], ((u - 1) >> 1) & 1)) {
                    ok = false;
                    break;
                }
            }
            float pr[32];
#pragma unroll
            for (int h = 0; h < 32; ++h) {
                const float ms = m[h] == -INFINITY ? 0.f : m[h];
                pr[h] = exp2f(x[h] - ms);
                l[h] += pr[h];
            }
            uint8_t *prow = p_buf;
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
                *reinterpret_cast<uint4 *>(prow + ptx::sw128_offset(r, half * 4 + c4)) = pack8(pr + 8 * c4);
            ptx::fence_proxy_async();
            ptx::mbar_arrive(&p_full[buf]);
        }
        if (!ok) *abort_flag = 1;
        // ---- the split's results: row sums, running max, unnormalised O ----
        if (ok && !*abort_flag &&
            ptx::mbar_wait(&pv_done[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1)) {
            ptx::tc_fence_after();
            // row sums over the 128 rows; the P buffers are free now (every PV is done)
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
                    if (h < a.H) {
                        a.part_m[pidx0 + h] = m[lane];
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
    }
    __syncthreads();
    if (warp == kAtMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, Cfg::TMEM_COLS);
    }
}

}  // namespace lca

// lca.cu -- the C ABI of liblca (declared in include/lca.h): host-side validation, work
// planning and kernel launches.  The library is built as one translation unit so that the
// device error word is a single object per device.
#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cmath>
#include <string>
#include <utility>

#include "../../include/lca.h"
#include "common.cuh"
#include "compress.cuh"
#include "quant.cuh"
#include "topk.cuh"
#include "indexer_tc.cuh"
#include "attend_common.cuh"
#include "attend_tc.cuh"
#include "gemv.cuh"
#include "gemm_tc.cuh"
#include "mhc.cuh"

using namespace lca;

namespace {

thread_local std::string t_last_error;

lca_status fail(lca_status s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return s;
}

lca_status ok() {
    t_last_error.clear();
    return LCA_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

lca_status check_launch(const char *what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(LCA_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
    return LCA_OK;
}

// Launch with programmatic dependent launch allowed: the kernel may be scheduled while the
// previous kernel in the stream runs; it waits for it (pdl_wait) before touching memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

int device_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
    return n;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// A bf16 tensor map of rank 2 or 3 (dims innermost first, strides in bytes for dims 1..),
// tiled boxes with the given swizzle; out-of-range elements read as zero.
bool make_tensor_map(CUtensorMap *map, const void *base, int rank, const uint64_t *dims, const uint64_t *strides,
                     const uint32_t *box, CUtensorMapSwizzle swizzle,
                     CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t gd[3], gs[2];
    cuuint32_t bd[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bd[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
    CUresult r = enc(map, dtype, rank, const_cast<void *>(base), gd, gs, bd, es,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

#define LCA_REQUIRE(cond, status, ...) \
    do {                                \
        if (!(cond)) return fail(status, __VA_ARGS__); \
    } while (0)

// theta_d / (2 pi) for d < R/2 in unsigned 0.64 fixed point (see RopeTable), in long double.
RopeTable make_rope_table(int rope_dims, float rope_base) {
    RopeTable t;
    const long double two_pi = 6.283185307179586476925286766559005768L;
    for (int d = 0; d < kMaxRopePairs; ++d) {
        t.f[d] = 0;
        if (rope_dims > 0 && d < rope_dims / 2) {
            const long double theta = powl((long double)rope_base, -2.0L * d / (long double)rope_dims);
            const long double frac = theta / two_pi;                       // < 1
            t.f[d] = (uint64_t)(frac * 18446744073709551616.0L);           // * 2^64
        }
    }
    return t;
}

RowNormRope make_nr(const lca_attn_params *p, const float *gamma, int apply_rope) {
    RowNormRope nr;
    nr.gamma = gamma;
    nr.eps = p->rms_eps;
    nr.rope_dims = apply_rope ? p->rope_dims : 0;
    nr.rope = make_rope_table(nr.rope_dims, p->rope_base);
    return nr;
}

lca_status compress_impl(const char *name, bool overlap, const lca_compress_variant *variant,
                         const lca_attn_params *p, int batch, int width,
                         const lca_bf16 *tok_v, int64_t tok_v_bs, int n_tok, const float *tok_z,
                         int64_t tok_z_bs, const int32_t *tok_pos0, const float *pos_bias,
                         const float *gamma, int apply_rope, const int32_t *first_entry, int n_new,
                         void *cache, int64_t cache_bs, int64_t cache_rows, cudaStream_t stream) {
    const bool pc = variant && variant->per_channel, fp8 = variant && variant->e4m3;
    LCA_REQUIRE(p, LCA_ERR_INVALID_ARG, "%s: params is NULL", name);
    LCA_REQUIRE(batch > 0 && n_tok > 0 && n_new >= 0, LCA_ERR_INVALID_ARG,
                "%s: batch (%d) and n_tok (%d) must be positive, n_new (%d) >= 0", name, batch, n_tok, n_new);
    LCA_REQUIRE(width >= 8 && width <= kMaxRowWidth && width % 8 == 0, LCA_ERR_UNSUPPORTED,
                "%s: width %d must be a multiple of 8 in [8, %d]", name, width, kMaxRowWidth);
    LCA_REQUIRE(p->ratio > 0, LCA_ERR_INVALID_ARG, "%s: ratio must be positive", name);
    const int span = overlap ? 2 * p->ratio : p->ratio;
    LCA_REQUIRE(span <= kMaxSpan, LCA_ERR_UNSUPPORTED, "%s: window of %d tokens exceeds %d", name, span, kMaxSpan);
    LCA_REQUIRE(tok_v && tok_z && tok_pos0 && pos_bias && first_entry && cache, LCA_ERR_INVALID_ARG,
                "%s: a required pointer is NULL", name);
    LCA_REQUIRE(aligned16(tok_v) && (fp8 ? reinterpret_cast<uintptr_t>(cache) % 8 == 0 : aligned16(cache)),
                LCA_ERR_INVALID_ARG, "%s: tok_v must be 16-byte aligned, cache 16 (bf16) or 8 (e4m3)", name);
    LCA_REQUIRE(tok_v_bs % 8 == 0 && cache_bs % 8 == 0, LCA_ERR_INVALID_ARG,
                "%s: batch strides must be multiples of 8 elements", name);
    const int64_t z_row = pc ? (int64_t)width : 1;           // logits per token
    LCA_REQUIRE(batch == 1 || (tok_v_bs >= (int64_t)n_tok * width && tok_z_bs >= n_tok * z_row &&
                               cache_bs >= cache_rows * width),
                LCA_ERR_INVALID_ARG, "%s: batch strides smaller than one sequence", name);
    if (pc)
        LCA_REQUIRE(aligned16(tok_z) && aligned16(pos_bias) && tok_z_bs % 4 == 0, LCA_ERR_INVALID_ARG,
                    "%s: per-channel tok_z and pos_bias must be 16-byte aligned, tok_z stride %% 4", name);
    if (fp8)
        LCA_REQUIRE(variant->cache_scale && (batch == 1 || variant->scale_batch_stride >= cache_rows),
                    LCA_ERR_INVALID_ARG, "%s: e4m3 cache needs cache_scale with a stride >= cache_rows", name);
    LCA_REQUIRE(cache_rows > 0, LCA_ERR_INVALID_ARG, "%s: cache_rows must be positive", name);
    if (apply_rope)
        LCA_REQUIRE(p->rope_dims > 0 && p->rope_dims % 2 == 0 && p->rope_dims <= width &&
                        p->rope_dims <= 2 * kMaxRopePairs && p->rope_base > 1.0f,
                    LCA_ERR_INVALID_ARG, "%s: rope_dims %d must be even, <= width and <= %d; base > 1", name,
                    p->rope_dims, 2 * kMaxRopePairs);
    if (n_new == 0) return ok();
    CompressArgs a;
    a.span = span;
    a.stride = p->ratio;
    a.width = width;
    a.tok_v = reinterpret_cast<const __nv_bfloat16 *>(tok_v);
    a.tok_v_bs = tok_v_bs;
    a.n_tok = n_tok;
    a.tok_z = tok_z;
    a.tok_z_bs = tok_z_bs;
    a.tok_pos0 = tok_pos0;
    a.bias = pos_bias;
    a.first_entry = first_entry;
    a.n_new = n_new;
    a.cache = fp8 ? nullptr : reinterpret_cast<__nv_bfloat16 *>(cache);
    a.cache8 = fp8 ? reinterpret_cast<uint8_t *>(cache) : nullptr;
    a.cache_scale = fp8 ? variant->cache_scale : nullptr;
    a.scale_bs = fp8 ? variant->scale_batch_stride : 0;
    a.cache_bs = cache_bs;
    a.cache_rows = cache_rows;
    a.nr = make_nr(p, gamma, apply_rope);
    const int threads = compress_threads(width, a.span);
    const size_t smem = compress_smem(threads, pc);
    auto launch = [&](auto kern) {
        if (smem > 48 * 1024) cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        launch_pdl(kern, dim3(n_new, batch), dim3(threads), smem, stream, a);
    };
    if (pc) fp8 ? launch(compress_kernel<true, true>) : launch(compress_kernel<true, false>);
    else fp8 ? launch(compress_kernel<false, true>) : launch(compress_kernel<false, false>);
    lca_status s = check_launch(name);
    return s == LCA_OK ? ok() : s;
}

// ---- attention planning ----
struct AttendPlan {
    int splits;
    int64_t units;
    size_t part_bytes;       // O partials
    size_t ml_bytes;         // m and l partials
    size_t img_bytes;        // per-query hi / lo images of the prepared query
    size_t total;
};

constexpr int kPlanTileRows = kAtTile;

// Split-K plan: one CTA per (query, split) and one CTA per SM, so a query gets as many splits
// as keep all SMs busy in one wave (and never more splits than tiles).  The byte counts cannot
// wrap: attend_validate bounds batch * n_q by kMaxAttendUnits, so the largest total is below
// 2^31 units x 128 splits x 64 heads x 512 x 4 bytes < 2^63 (the same bound keeps
// *_attend_workspace from returning a wrapped size).
constexpr int64_t kMaxAttendUnits = (int64_t)1 << 31;
AttendPlan plan_attend(const lca_attn_params *p, int batch, int n_q, int64_t max_rows) {
    AttendPlan pl;
    pl.units = (int64_t)batch * n_q;
    const int64_t tiles = ceil_div64(max_rows, kPlanTileRows);
    const int sms = device_sm_count();
    int64_t s = sms / pl.units;
    if (s > tiles) s = tiles;
    if (s < 1) s = 1;
    if (s > kMaxSplits) s = kMaxSplits;
    pl.splits = (int)s;
    pl.part_bytes = (size_t)pl.units * pl.splits * p->heads * p->head_dim * sizeof(float);
    pl.ml_bytes = (size_t)pl.units * pl.splits * p->heads * sizeof(float);
    pl.img_bytes = (size_t)pl.units * (p->head_dim / 128) * kQChunkBytes;
    pl.total = pl.part_bytes + 2 * ((pl.ml_bytes + 255) & ~(size_t)255) + pl.img_bytes;
    return pl;
}

lca_status attend_validate(const char *name, const lca_attn_params *p, int batch, int n_q) {
    LCA_REQUIRE(p, LCA_ERR_INVALID_ARG, "%s: params is NULL", name);
    LCA_REQUIRE(batch > 0 && n_q > 0, LCA_ERR_INVALID_ARG, "%s: batch and n_q must be positive", name);
    LCA_REQUIRE((int64_t)batch * n_q < kMaxAttendUnits, LCA_ERR_UNSUPPORTED,
                "%s: batch * n_q = %lld queries, at most 2^31 - 1 per call", name, (long long)batch * n_q);
    LCA_REQUIRE(p->head_dim == 128 || p->head_dim == 256 || p->head_dim == 512, LCA_ERR_UNSUPPORTED,
                "%s: head_dim %d not in {128, 256, 512}", name, p->head_dim);
    LCA_REQUIRE(p->heads >= 1 && p->heads <= 64, LCA_ERR_UNSUPPORTED, "%s: heads %d not in [1, 64]", name, p->heads);
    const int epl = p->head_dim / 32;
    LCA_REQUIRE(p->rope_dims >= 0 && p->rope_dims <= p->head_dim && p->rope_dims % 2 == 0 &&
                    (p->rope_dims / 2) % epl == 0 && p->rope_dims <= 2 * kMaxRopePairs &&
                    (p->rope_dims == 0 || p->rope_base > 1.0f),
                LCA_ERR_UNSUPPORTED, "%s: rope_dims %d must be even, <= c and R/2 a multiple of c/32", name,
                p->rope_dims);
    LCA_REQUIRE(p->window >= 1 && p->window <= 4096, LCA_ERR_UNSUPPORTED, "%s: window %d not in [1, 4096]", name,
                p->window);
    return LCA_OK;
}

// What an attention call launches: the query preparation and the attention (the usual call),
// the attention alone (the query image is already in the workspace), or the preparation alone.
enum AttendMode { kAttendAll = 0, kAttendPrepared = 1, kAttendPrepareOnly = 2 };

lca_status attend_impl(const char *name, const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q,
                       const float *gamma_q, const int32_t *q_pos, const lca_bf16 *kv, int64_t kv_bs,
                       int64_t cache_rows, const int32_t *idx, const lca_bf16 *win, int64_t win_bs,
                       int win_cap, const float *sink, lca_bf16 *out, float *lse, void *ws, size_t ws_bytes,
                       cudaStream_t stream, AttendMode mode = kAttendAll, const uint8_t *kv8 = nullptr,
                       const float *kv_scale = nullptr, int64_t ks_bs = 0) {
    lca_status st = attend_validate(name, p, batch, n_q);
    if (st != LCA_OK) return st;
    const bool csa = idx != nullptr;
    const bool e4m3 = kv8 != nullptr;        // the compressed rows come from an e4m3 cache
    if (csa) LCA_REQUIRE(p->topk >= 1, LCA_ERR_INVALID_ARG, "%s: topk must be positive", name);
    else LCA_REQUIRE(p->ratio >= 1, LCA_ERR_INVALID_ARG, "%s: ratio must be positive", name);
    const void *kvp = e4m3 ? static_cast<const void *>(kv8) : static_cast<const void *>(kv);
    LCA_REQUIRE(q && gamma_q && q_pos && kvp && win && sink && out, LCA_ERR_INVALID_ARG,
                "%s: a required pointer is NULL", name);
    LCA_REQUIRE(aligned16(q) && aligned16(kvp) && aligned16(win) && aligned16(out), LCA_ERR_INVALID_ARG,
                "%s: q, kv_cache, win_kv and out must be 16-byte aligned", name);
    if (e4m3) {
        LCA_REQUIRE(p->head_dim == 512, LCA_ERR_UNSUPPORTED, "%s: e4m3 rows need head_dim 512", name);
        LCA_REQUIRE(kv_scale && reinterpret_cast<uintptr_t>(kv_scale) % 4 == 0 &&
                        (batch == 1 || ks_bs >= cache_rows),
                    LCA_ERR_INVALID_ARG, "%s: kv_scale (4-byte aligned, stride >= cache_rows) is required", name);
    }
    LCA_REQUIRE(kv_bs % 8 == 0 && win_bs % 8 == 0, LCA_ERR_INVALID_ARG,
                "%s: batch strides must be multiples of 8 elements", name);
    LCA_REQUIRE(cache_rows > 0, LCA_ERR_INVALID_ARG, "%s: cache_rows must be positive", name);
    LCA_REQUIRE(win_cap >= p->window, LCA_ERR_INVALID_ARG, "%s: win_cap %d < window %d", name, win_cap, p->window);
    LCA_REQUIRE(batch == 1 || (kv_bs >= cache_rows * p->head_dim && win_bs >= (int64_t)win_cap * p->head_dim &&
                               kv_bs % p->head_dim == 0 && win_bs % p->head_dim == 0),
                LCA_ERR_INVALID_ARG, "%s: batch strides must cover a sequence and be multiples of head_dim", name);
    LCA_REQUIRE((int64_t)(batch - 1) * (kv_bs / p->head_dim) + cache_rows < ((int64_t)1 << 31) &&
                    (int64_t)(batch - 1) * (win_bs / p->head_dim) + win_cap < ((int64_t)1 << 31),
                LCA_ERR_UNSUPPORTED, "%s: caches exceed 2^31 rows", name);
    const int64_t max_rows = (csa ? p->topk : cache_rows) + p->window;
    AttendPlan pl = plan_attend(p, batch, n_q, max_rows);
    LCA_REQUIRE(ws && aligned16(ws) && ws_bytes >= pl.total, LCA_ERR_WORKSPACE,
                "%s: workspace of %zu bytes (16-byte aligned) needed, got %zu", name, pl.total, ws_bytes);
    AttendArgs a;
    a.H = p->heads;
    a.C = p->head_dim;
    a.R = p->rope_dims;
    a.rope = make_rope_table(p->rope_dims, p->rope_base);
    a.eps = p->rms_eps;
    const float scale = p->softmax_scale > 0.f ? p->softmax_scale : 1.0f / sqrtf((float)p->head_dim);
    a.scale_log2 = scale * kLog2e;
    a.W = p->window;
    a.ratio = p->ratio;
    a.n_idx = csa ? p->topk : 0;
    a.n_q = n_q;
    a.splits = pl.splits;
    a.q = reinterpret_cast<const __nv_bfloat16 *>(q);
    a.gamma_q = gamma_q;
    a.q_pos = q_pos;
    a.kv = e4m3 ? nullptr : reinterpret_cast<const __nv_bfloat16 *>(kv);
    a.kv_bs = kv_bs;
    a.kv_scale = kv_scale;
    a.ks_bs = ks_bs;
    a.cache_rows = cache_rows;
    a.idx = idx;
    a.win = reinterpret_cast<const __nv_bfloat16 *>(win);
    a.win_bs = win_bs;
    a.win_cap = win_cap;
    a.sink = sink;
    char *w = static_cast<char *>(ws);
    a.part_o = reinterpret_cast<float *>(w);
    a.part_m = reinterpret_cast<float *>(w + pl.part_bytes);
    a.part_l = reinterpret_cast<float *>(w + pl.part_bytes + ((pl.ml_bytes + 255) & ~(size_t)255));
    a.q_img = reinterpret_cast<uint8_t *>(w + pl.part_bytes + 2 * ((pl.ml_bytes + 255) & ~(size_t)255));
    a.out = reinterpret_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    LCA_REQUIRE(pl.units <= 0x7fffffff, LCA_ERR_UNSUPPORTED, "%s: too many queries", name);
    dim3 grid((unsigned)pl.units, pl.splits);
    // tensor maps: the caches as 2D [rows, c] views (sequence b starts at row b * bs / c)
    const int C = p->head_dim;
    const uint64_t kv_rows = (uint64_t)(batch - 1) * (uint64_t)(kv_bs / C) + (uint64_t)cache_rows;
    const uint64_t win_rows = (uint64_t)(batch - 1) * (uint64_t)(win_bs / C) + (uint64_t)win_cap;
    const uint64_t dims_kv[2] = {(uint64_t)C, kv_rows}, dims_win[2] = {(uint64_t)C, win_rows};
    const uint64_t row_bytes[1] = {(uint64_t)C * 2};
    const uint32_t box_tile[2] = {64, (uint32_t)kAtTile}, box_row[2] = {64, 1};
    // e4m3 rows: 128 codes (128 bytes) per box row
    const uint64_t row_bytes8[1] = {(uint64_t)C};
    const uint32_t box_tile8[2] = {128, (uint32_t)kAtTile}, box_row8[2] = {128, 1};
    CUtensorMap kv_tile_map, kv_row_map, win_row_map;
    const bool maps_ok =
        (e4m3 ? make_tensor_map(&kv_tile_map, kvp, 2, dims_kv, row_bytes8, box_tile8, CU_TENSOR_MAP_SWIZZLE_128B,
                                CU_TENSOR_MAP_DATA_TYPE_UINT8) &&
                    make_tensor_map(&kv_row_map, kvp, 2, dims_kv, row_bytes8, box_row8, CU_TENSOR_MAP_SWIZZLE_128B,
                                    CU_TENSOR_MAP_DATA_TYPE_UINT8)
              : make_tensor_map(&kv_tile_map, kvp, 2, dims_kv, row_bytes, box_tile, CU_TENSOR_MAP_SWIZZLE_128B) &&
                    make_tensor_map(&kv_row_map, kvp, 2, dims_kv, row_bytes, box_row, CU_TENSOR_MAP_SWIZZLE_128B)) &&
        make_tensor_map(&win_row_map, win, 2, dims_win, row_bytes, box_row, CU_TENSOR_MAP_SWIZZLE_128B);
    if (!maps_ok) return fail(LCA_ERR_CUDA, "%s: tensor map rejected by the driver", name);
    if (mode != kAttendPrepared) {
        const dim3 prep_grid((unsigned)pl.units, kQImgHeads / kQPrepHeads);
        switch (C) {
        case 128: launch_pdl(q_prep_kernel<128>, prep_grid, dim3(32 * kQPrepHeads), 0, stream, a); break;
        case 256: launch_pdl(q_prep_kernel<256>, prep_grid, dim3(32 * kQPrepHeads), 0, stream, a); break;
        default: launch_pdl(q_prep_kernel<512>, prep_grid, dim3(32 * kQPrepHeads), 0, stream, a); break;
        }
        st = check_launch(name);
        if (st != LCA_OK) return st;
        if (mode == kAttendPrepareOnly) return ok();
    }
    if (e4m3) {
        cudaFuncSetAttribute(attend_tc_kernel<512, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AttendTcConfig<512>::SMEM_BYTES);
        launch_pdl(attend_tc_kernel<512, true>, grid, dim3(kAtThreads), AttendTcConfig<512>::SMEM_BYTES, stream,
                   kv_tile_map, kv_row_map, win_row_map, a);
    } else
    switch (C) {
    case 128:
        cudaFuncSetAttribute(attend_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AttendTcConfig<128>::SMEM_BYTES);
        launch_pdl(attend_tc_kernel<128>, grid, dim3(kAtThreads), AttendTcConfig<128>::SMEM_BYTES, stream, kv_tile_map,
                   kv_row_map, win_row_map, a);
        break;
    case 256:
        cudaFuncSetAttribute(attend_tc_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AttendTcConfig<256>::SMEM_BYTES);
        launch_pdl(attend_tc_kernel<256>, grid, dim3(kAtThreads), AttendTcConfig<256>::SMEM_BYTES, stream, kv_tile_map,
                   kv_row_map, win_row_map, a);
        break;
    default:
        cudaFuncSetAttribute(attend_tc_kernel<512>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             AttendTcConfig<512>::SMEM_BYTES);
        launch_pdl(attend_tc_kernel<512>, grid, dim3(kAtThreads), AttendTcConfig<512>::SMEM_BYTES, stream, kv_tile_map,
                   kv_row_map, win_row_map, a);
        break;
    }
    st = check_launch(name);
    if (st != LCA_OK) return st;
    launch_pdl(combine_kernel, dim3((unsigned)pl.units, p->heads), dim3(kCombineThreads), 0, stream, a);
    st = check_launch(name);
    return st == LCA_OK ? ok() : st;
}

lca_status indexer_validate(const char *name, const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q_idx,
                            const float *w_idx, const lca_bf16 *k_cache, int64_t k_bs, int64_t cache_rows,
                            const int32_t *q_pos) {
    LCA_REQUIRE(p, LCA_ERR_INVALID_ARG, "%s: params is NULL", name);
    LCA_REQUIRE(batch > 0 && n_q > 0 && cache_rows > 0 && cache_rows < INT32_MAX, LCA_ERR_INVALID_ARG,
                "%s: batch, n_q and cache_rows must be positive, cache_rows < 2^31", name);
    LCA_REQUIRE(p->ratio >= 1, LCA_ERR_INVALID_ARG, "%s: ratio must be positive", name);
    LCA_REQUIRE((p->idx_dim == 128 && p->idx_heads == 64) || (p->idx_dim == 64 && p->idx_heads == 32) ||
                    (p->idx_dim == 32 && p->idx_heads == 4),
                LCA_ERR_UNSUPPORTED, "%s: indexer (heads %d, dim %d) not in {(64, 128), (32, 64), (4, 32)}", name,
                p->idx_heads, p->idx_dim);
    LCA_REQUIRE(q_idx && w_idx && k_cache && q_pos, LCA_ERR_INVALID_ARG, "%s: a required pointer is NULL", name);
    LCA_REQUIRE(aligned16(q_idx) && aligned16(k_cache), LCA_ERR_INVALID_ARG,
                "%s: q_idx and k_cache must be 16-byte aligned", name);
    LCA_REQUIRE(k_bs % 8 == 0 && (batch == 1 || k_bs >= cache_rows * p->idx_dim), LCA_ERR_INVALID_ARG,
                "%s: bad k_batch_stride", name);
    return LCA_OK;
}

template <int DI, int HI, int QPT, bool FUSE = false, bool FP8 = false>
lca_status indexer_tc_launch(int batch, int n_q, const void *q_idx, const void *k_cache, int64_t k_bs,
                             IndexerTcArgs &a, cudaStream_t stream) {
    using Cfg = IndexerTcConfig<DI, HI, QPT, FUSE, FP8>;
    const CUtensorMapSwizzle sw = Cfg::ROWB == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    constexpr uint64_t E = Cfg::ESZ;
    CUtensorMap kmap, qmap;
    const uint64_t kd[3] = {(uint64_t)DI, (uint64_t)a.cache_rows, (uint64_t)batch};
    const uint64_t ks[2] = {(uint64_t)DI * E, (uint64_t)k_bs * E};
    const uint32_t kb[3] = {(uint32_t)Cfg::BOX, 128u, 1u};
    if (!make_tensor_map(&kmap, k_cache, 3, kd, ks, kb, sw, dt))
        return fail(LCA_ERR_CUDA, "csa_indexer_scores: key tensor map rejected by the driver");
    const uint64_t qd[2] = {(uint64_t)DI, (uint64_t)batch * n_q * HI};
    const uint64_t qs[1] = {(uint64_t)DI * E};
    const uint32_t qb[2] = {(uint32_t)Cfg::BOX, (uint32_t)Cfg::N};
    if (!make_tensor_map(&qmap, q_idx, 2, qd, qs, qb, sw, dt))
        return fail(LCA_ERR_CUDA, "csa_indexer_scores: query tensor map rejected by the driver");
    CUtensorMap smap = kmap;                  // e4m3: the key scales, 128 per tile
    if (FP8) {
        const uint64_t sd[2] = {(uint64_t)a.cache_rows, (uint64_t)batch};
        const uint64_t ss[1] = {batch == 1 ? (uint64_t)((a.cache_rows * 4 + 15) / 16 * 16) : (uint64_t)a.ks_bs * 4};
        const uint32_t sb[2] = {128u, 1u};
        if (!make_tensor_map(&smap, a.k_scale, 2, sd, ss, sb, CU_TENSOR_MAP_SWIZZLE_NONE,
                             CU_TENSOR_MAP_DATA_TYPE_FLOAT32))
            return fail(LCA_ERR_CUDA, "csa_indexer_scores_e4m3: key scale tensor map rejected by the driver");
    }
    a.groups = (n_q + QPT - 1) / QPT;
    a.tiles = (int)ceil_div64(a.cache_rows, 128);
    a.items = (int64_t)batch * a.groups * a.tiles;
    // the fused selection hands each CTA whole query groups
    const int grid = (int)std::min<int64_t>(FUSE ? (int64_t)batch * a.groups : a.items, device_sm_count());
    cudaFuncSetAttribute(indexer_tc_kernel<DI, HI, QPT, FUSE, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         Cfg::SMEM_BYTES);
    launch_pdl(indexer_tc_kernel<DI, HI, QPT, FUSE, FP8>, grid, dim3(Cfg::THREADS), Cfg::SMEM_BYTES, stream, kmap,
               qmap, smap, a);
    return check_launch(FUSE ? "csa_indexer_topk" : "csa_indexer_scores");
}

lca_status indexer_launch(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q_idx, const float *w_idx,
                          const lca_bf16 *k_cache, int64_t k_bs, int64_t cache_rows, const int32_t *q_pos,
                          float *scores, int64_t s_stride, cudaStream_t stream) {
    IndexerTcArgs a;
    a.n_q = n_q;
    a.ratio = p->ratio;
    a.cache_rows = cache_rows;
    a.w = w_idx;
    a.q_pos = q_pos;
    a.scores = scores;
    a.stride = s_stride;
    if (p->idx_dim == 128) {
        if (n_q == 1) return indexer_tc_launch<128, 64, 1>(batch, n_q, q_idx, k_cache, k_bs, a, stream);
        if (n_q == 2) return indexer_tc_launch<128, 64, 2>(batch, n_q, q_idx, k_cache, k_bs, a, stream);
        return indexer_tc_launch<128, 64, 4>(batch, n_q, q_idx, k_cache, k_bs, a, stream);
    }
    if (p->idx_dim == 64) {
        if (n_q == 1) return indexer_tc_launch<64, 32, 1>(batch, n_q, q_idx, k_cache, k_bs, a, stream);
        return indexer_tc_launch<64, 32, 8>(batch, n_q, q_idx, k_cache, k_bs, a, stream);
    }
    return indexer_tc_launch<32, 4, 4>(batch, n_q, q_idx, k_cache, k_bs, a, stream);
}

lca_status topk_launch(const lca_attn_params *p, int batch, int n_q, const float *scores, int64_t s_stride,
                       const int32_t *q_pos, int64_t max_entries, int32_t *out_idx, cudaStream_t stream) {
    TopkArgs a;
    a.scores = scores;
    a.row_stride = s_stride;
    a.q_pos = q_pos;
    a.ratio = p->ratio;
    a.max_entries = max_entries;
    a.k = p->topk;
    a.out = out_idx;
    const int64_t rows = (int64_t)batch * n_q;
    // CTAs per row: enough to cover the SMs when rows are few (decode), one otherwise
    int cl = (int)std::min<int64_t>(kTopkMaxCluster, std::max<int64_t>(1, device_sm_count() / rows));
    while (cl > 1 && (int64_t)cl * (cl - 1) >= max_entries) cl /= 2;   // slices of at least a few keys
    a.cl = cl;
    const int64_t slice = ((max_entries + cl - 1) / cl + 3) & ~(int64_t)3;
    const bool smem_keys = slice <= kTopkSmemKeys;
    const int smem = (int)topk_smem_bytes(smem_keys, slice);
    auto kern = smem_keys ? topk_kernel<true> : topk_kernel<false>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows * cl));
    cfg.blockDim = dim3(kTopkThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return fail(LCA_ERR_CUDA, "lca_topk: launch failed: %s", cudaGetErrorString(e));
    return check_launch("lca_topk");
}

lca_status indexer_e4m3_validate(const char *name, const lca_attn_params *p, int batch, int n_q, const uint8_t *q8,
                                 const float *q_scale, const float *w_idx, const uint8_t *k8, int64_t k_bs,
                                 const float *k_scale, int64_t ks_bs, int64_t cache_rows, const int32_t *q_pos) {
    LCA_REQUIRE(p, LCA_ERR_INVALID_ARG, "%s: params is NULL", name);
    LCA_REQUIRE(batch > 0 && n_q > 0 && cache_rows > 0 && cache_rows < INT32_MAX, LCA_ERR_INVALID_ARG,
                "%s: batch, n_q and cache_rows must be positive, cache_rows < 2^31", name);
    LCA_REQUIRE(p->ratio >= 1, LCA_ERR_INVALID_ARG, "%s: ratio must be positive", name);
    LCA_REQUIRE(p->idx_dim == 128 && p->idx_heads == 64, LCA_ERR_UNSUPPORTED,
                "%s: e4m3 indexer supports 64 heads of dim 128 (got %d, %d)", name, p->idx_heads, p->idx_dim);
    LCA_REQUIRE(q8 && q_scale && w_idx && k8 && k_scale && q_pos, LCA_ERR_INVALID_ARG,
                "%s: a required pointer is NULL", name);
    LCA_REQUIRE(aligned16(q8) && aligned16(k8), LCA_ERR_INVALID_ARG, "%s: q_idx8 and k_cache8 must be 16-byte aligned",
                name);
    LCA_REQUIRE(k_bs % 16 == 0 && (batch == 1 || (k_bs >= cache_rows * p->idx_dim && ks_bs >= cache_rows &&
                                                   ks_bs % 4 == 0)),
                LCA_ERR_INVALID_ARG, "%s: bad k_batch_stride / k_scale_batch_stride (%% 4)", name);
    LCA_REQUIRE(aligned16(k_scale), LCA_ERR_INVALID_ARG, "%s: k_scale must be 16-byte aligned", name);
    return LCA_OK;
}

IndexerTcArgs indexer_e4m3_args(const lca_attn_params *p, int n_q, const float *q_scale, const float *w_idx,
                                const float *k_scale, int64_t ks_bs, int64_t cache_rows, const int32_t *q_pos) {
    IndexerTcArgs a = {};
    a.n_q = n_q;
    a.ratio = p->ratio;
    a.cache_rows = cache_rows;
    a.w = w_idx;
    a.q_pos = q_pos;
    a.q_scale = q_scale;
    a.k_scale = k_scale;
    a.ks_bs = ks_bs;
    return a;
}

lca_status indexer_e4m3_scores_launch(const lca_attn_params *p, int batch, int n_q, const uint8_t *q8,
                                      const float *q_scale, const float *w_idx, const uint8_t *k8, int64_t k_bs,
                                      const float *k_scale, int64_t ks_bs, int64_t cache_rows, const int32_t *q_pos,
                                      float *scores, int64_t s_stride, cudaStream_t stream) {
    IndexerTcArgs a = indexer_e4m3_args(p, n_q, q_scale, w_idx, k_scale, ks_bs, cache_rows, q_pos);
    a.scores = scores;
    a.stride = s_stride;
    if (n_q == 1) return indexer_tc_launch<128, 64, 1, false, true>(batch, n_q, q8, k8, k_bs, a, stream);
    if (n_q == 2) return indexer_tc_launch<128, 64, 2, false, true>(batch, n_q, q8, k8, k_bs, a, stream);
    return indexer_tc_launch<128, 64, 4, false, true>(batch, n_q, q8, k8, k_bs, a, stream);
}

size_t indexer_ws_bytes(int batch, int n_q, int64_t cache_rows) {
    const int64_t stride = (cache_rows + 3) & ~(int64_t)3;
    return (size_t)batch * n_q * stride * sizeof(float);
}

// Whether csa_indexer_topk selects inside the indexer (four queries per tile: d_I = 128 with
// H_I = 64 and n_q >= 3; k within the streaming selection's limit).
bool indexer_fused(const lca_attn_params *p, int n_q) {
    return p->idx_dim == 128 && p->idx_heads == 64 && n_q >= 3 && p->topk >= 1 && p->topk <= kStMaxK;
}

// The fused path's candidate buffers: per CTA, two buffers per warp group and query.
size_t indexer_cand_bytes(int batch, int n_q) {
    const int64_t groups = (int64_t)batch * ((n_q + 3) / 4);
    const int64_t grid = std::min<int64_t>(groups, device_sm_count());
    return (size_t)grid * IndexerTcConfig<128, 64, 4, true>::CAND_PER_CTA * sizeof(uint2);
}

}  // namespace

extern "C" {

const char *lca_version(void) { return "lca 0.1 (sm_103a)"; }

const char *lca_status_string(lca_status s) {
    switch (s) {
    case LCA_OK: return "ok";
    case LCA_ERR_INVALID_ARG: return "invalid argument";
    case LCA_ERR_UNSUPPORTED: return "unsupported shape";
    case LCA_ERR_WORKSPACE: return "workspace too small";
    case LCA_ERR_CUDA: return "CUDA error";
    case LCA_ERR_TIMEOUT: return "kernel wait timed out";
    case LCA_ERR_DEVICE: return "device-side check failed";
    }
    return "unknown status";
}

const char *lca_last_error(void) { return t_last_error.c_str(); }

lca_status lca_test_hooks(long long wait_limit_cycles, int attend_skip_tile) {
    const long long limit = wait_limit_cycles > 0 ? wait_limit_cycles : 2000000000LL;
    LCA_REQUIRE(attend_skip_tile != 0, LCA_ERR_INVALID_ARG, "lca_test_hooks: the skipped tile must be 1 or later");
    const int skip = attend_skip_tile >= 1 ? attend_skip_tile : -1;
    cudaError_t e = cudaMemcpyToSymbol(g_wait_limit_cycles, &limit, sizeof limit);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_test_skip_tile, &skip, sizeof skip);
    if (e != cudaSuccess) return fail(LCA_ERR_CUDA, "lca_test_hooks: %s", cudaGetErrorString(e));
    return ok();
}

lca_status lca_device_error(cudaStream_t stream, uint32_t *word) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return fail(LCA_ERR_CUDA, "lca_device_error: %s", cudaGetErrorString(e));
    unsigned int w = 0, zero = 0;
    e = cudaMemcpyFromSymbol(&w, g_error_word, sizeof w);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof zero);
    if (e != cudaSuccess) return fail(LCA_ERR_CUDA, "lca_device_error: %s", cudaGetErrorString(e));
    if (word) *word = w;
    if (w & LCA_DEVERR_TIMEOUT) return fail(LCA_ERR_TIMEOUT, "a bounded wait inside a kernel ran out (0x%x)", w);
    if (w) return fail(LCA_ERR_DEVICE, "device-side check failed (0x%x)", w);
    return ok();
}

lca_status csa_compress_kv(const lca_attn_params *p, int batch, int width, const lca_bf16 *tok_v,
                           int64_t tok_v_batch_stride, int n_tok, const float *tok_z, int64_t tok_z_batch_stride,
                           const int32_t *tok_pos0, const float *pos_bias, const float *gamma, int apply_rope,
                           const int32_t *first_entry, int n_new, lca_bf16 *cache, int64_t cache_batch_stride,
                           int64_t cache_rows, cudaStream_t stream) {
    return compress_impl("csa_compress_kv", true, nullptr, p, batch, width, tok_v, tok_v_batch_stride, n_tok, tok_z,
                         tok_z_batch_stride, tok_pos0, pos_bias, gamma, apply_rope, first_entry, n_new, cache,
                         cache_batch_stride, cache_rows, stream);
}

lca_status hca_compress_kv(const lca_attn_params *p, int batch, int width, const lca_bf16 *tok_v,
                           int64_t tok_v_batch_stride, int n_tok, const float *tok_z, int64_t tok_z_batch_stride,
                           const int32_t *tok_pos0, const float *pos_bias, const float *gamma, int apply_rope,
                           const int32_t *first_entry, int n_new, lca_bf16 *cache, int64_t cache_batch_stride,
                           int64_t cache_rows, cudaStream_t stream) {
    return compress_impl("hca_compress_kv", false, nullptr, p, batch, width, tok_v, tok_v_batch_stride, n_tok, tok_z,
                         tok_z_batch_stride, tok_pos0, pos_bias, gamma, apply_rope, first_entry, n_new, cache,
                         cache_batch_stride, cache_rows, stream);
}

lca_status csa_compress_kv_ex(const lca_attn_params *p, const lca_compress_variant *variant, int batch, int width,
                              const lca_bf16 *tok_v, int64_t tok_v_batch_stride, int n_tok, const float *tok_z,
                              int64_t tok_z_batch_stride, const int32_t *tok_pos0, const float *pos_bias,
                              const float *gamma, int apply_rope, const int32_t *first_entry, int n_new, void *cache,
                              int64_t cache_batch_stride, int64_t cache_rows, cudaStream_t stream) {
    LCA_REQUIRE(variant, LCA_ERR_INVALID_ARG, "csa_compress_kv_ex: variant is NULL");
    return compress_impl("csa_compress_kv_ex", true, variant, p, batch, width, tok_v, tok_v_batch_stride, n_tok,
                         tok_z, tok_z_batch_stride, tok_pos0, pos_bias, gamma, apply_rope, first_entry, n_new, cache,
                         cache_batch_stride, cache_rows, stream);
}

lca_status hca_compress_kv_ex(const lca_attn_params *p, const lca_compress_variant *variant, int batch, int width,
                              const lca_bf16 *tok_v, int64_t tok_v_batch_stride, int n_tok, const float *tok_z,
                              int64_t tok_z_batch_stride, const int32_t *tok_pos0, const float *pos_bias,
                              const float *gamma, int apply_rope, const int32_t *first_entry, int n_new, void *cache,
                              int64_t cache_batch_stride, int64_t cache_rows, cudaStream_t stream) {
    LCA_REQUIRE(variant, LCA_ERR_INVALID_ARG, "hca_compress_kv_ex: variant is NULL");
    return compress_impl("hca_compress_kv_ex", false, variant, p, batch, width, tok_v, tok_v_batch_stride, n_tok,
                         tok_z, tok_z_batch_stride, tok_pos0, pos_bias, gamma, apply_rope, first_entry, n_new, cache,
                         cache_batch_stride, cache_rows, stream);
}

lca_status lca_quantize_rows_e4m3(const lca_bf16 *x, int64_t rows, int width, uint8_t *q, float *scale,
                                  cudaStream_t stream) {
    const char *name = "lca_quantize_rows_e4m3";
    LCA_REQUIRE(x && q && scale, LCA_ERR_INVALID_ARG, "%s: a required pointer is NULL", name);
    LCA_REQUIRE(rows >= 0 && width >= 8 && width <= 32 * kQuantMaxChunks * 8 && width % 8 == 0, LCA_ERR_INVALID_ARG,
                "%s: width %d must be a multiple of 8 in [8, %d], rows >= 0", name, width, 32 * kQuantMaxChunks * 8);
    LCA_REQUIRE(aligned16(x) && reinterpret_cast<uintptr_t>(q) % 8 == 0, LCA_ERR_INVALID_ARG,
                "%s: x must be 16-byte aligned and q 8-byte aligned", name);
    if (rows == 0) return ok();
    LCA_REQUIRE(ceil_div64(rows, kQuantWarps) <= INT32_MAX, LCA_ERR_UNSUPPORTED, "%s: too many rows", name);
    QuantArgs a;
    a.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    a.rows = rows;
    a.width = width;
    a.q = q;
    a.scale = scale;
    launch_pdl(quantize_rows_kernel, (int)ceil_div64(rows, kQuantWarps), dim3(32 * kQuantWarps), 0, stream, a);
    lca_status s = check_launch(name);
    return s == LCA_OK ? ok() : s;
}

lca_status lca_window_update(const lca_attn_params *p, int batch, const lca_bf16 *tok_v, int64_t tok_v_batch_stride,
                             int n_tok, const int32_t *tok_pos0, const float *gamma, lca_bf16 *win_kv,
                             int64_t win_batch_stride, int win_cap, cudaStream_t stream) {
    const char *name = "lca_window_update";
    LCA_REQUIRE(p, LCA_ERR_INVALID_ARG, "%s: params is NULL", name);
    const int width = p->head_dim;
    LCA_REQUIRE(batch > 0 && n_tok >= 0 && win_cap > 0, LCA_ERR_INVALID_ARG,
                "%s: batch and win_cap must be positive", name);
    LCA_REQUIRE(width >= 8 && width <= kMaxRowWidth && width % 8 == 0, LCA_ERR_UNSUPPORTED,
                "%s: head_dim %d unsupported", name, width);
    LCA_REQUIRE(tok_v && tok_pos0 && gamma && win_kv, LCA_ERR_INVALID_ARG, "%s: a required pointer is NULL", name);
    LCA_REQUIRE(aligned16(tok_v) && aligned16(win_kv) && tok_v_batch_stride % 8 == 0 && win_batch_stride % 8 == 0,
                LCA_ERR_INVALID_ARG, "%s: misaligned pointer or stride", name);
    LCA_REQUIRE(p->rope_dims >= 0 && p->rope_dims % 2 == 0 && p->rope_dims <= width &&
                    p->rope_dims <= 2 * kMaxRopePairs && (p->rope_dims == 0 || p->rope_base > 1.0f),
                LCA_ERR_INVALID_ARG, "%s: bad rope_dims / rope_base", name);
    if (n_tok == 0) return ok();
    WindowArgs a;
    a.width = width;
    a.tok_v = reinterpret_cast<const __nv_bfloat16 *>(tok_v);
    a.tok_v_bs = tok_v_batch_stride;
    a.n_tok = n_tok;
    a.tok_pos0 = tok_pos0;
    a.win = reinterpret_cast<__nv_bfloat16 *>(win_kv);
    a.win_bs = win_batch_stride;
    a.win_cap = win_cap;
    a.nr = make_nr(p, gamma, p->rope_dims > 0);
    launch_pdl(window_kernel, dim3(n_tok, batch), dim3(kRowThreads), 0, stream, a);
    lca_status s = check_launch(name);
    return s == LCA_OK ? ok() : s;
}

lca_status csa_indexer_scores(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q_idx,
                              const float *w_idx, const lca_bf16 *k_cache, int64_t k_batch_stride,
                              int64_t cache_rows, const int32_t *q_pos, float *scores, int64_t scores_stride,
                              cudaStream_t stream) {
    const char *name = "csa_indexer_scores";
    lca_status st = indexer_validate(name, p, batch, n_q, q_idx, w_idx, k_cache, k_batch_stride, cache_rows, q_pos);
    if (st != LCA_OK) return st;
    LCA_REQUIRE(scores && aligned16(scores) && scores_stride >= cache_rows && scores_stride % 4 == 0,
                LCA_ERR_INVALID_ARG, "%s: scores must be 16-byte aligned with a stride >= cache_rows, %% 4", name);
    st = indexer_launch(p, batch, n_q, q_idx, w_idx, k_cache, k_batch_stride, cache_rows, q_pos, scores,
                        scores_stride, stream);
    return st == LCA_OK ? ok() : st;
}

lca_status lca_topk(const lca_attn_params *p, int batch, int n_q, const float *scores, int64_t scores_stride,
                    const int32_t *q_pos, int64_t max_entries, int32_t *out_idx, cudaStream_t stream) {
    const char *name = "lca_topk";
    LCA_REQUIRE(p, LCA_ERR_INVALID_ARG, "%s: params is NULL", name);
    LCA_REQUIRE(batch > 0 && n_q > 0 && max_entries >= 0, LCA_ERR_INVALID_ARG, "%s: bad sizes", name);
    LCA_REQUIRE(p->topk >= 1 && p->ratio >= 1, LCA_ERR_INVALID_ARG, "%s: topk and ratio must be positive", name);
    LCA_REQUIRE(scores && q_pos && out_idx, LCA_ERR_INVALID_ARG, "%s: a required pointer is NULL", name);
    LCA_REQUIRE(aligned4(scores) && scores_stride >= max_entries, LCA_ERR_INVALID_ARG,
                "%s: scores_stride must be >= max_entries", name);
    lca_status st = topk_launch(p, batch, n_q, scores, scores_stride, q_pos, max_entries, out_idx, stream);
    return st == LCA_OK ? ok() : st;
}

size_t csa_indexer_workspace(const lca_attn_params *p, int batch, int n_q, int64_t cache_rows) {
    if (!p || batch <= 0 || n_q <= 0 || cache_rows <= 0) return 0;
    return indexer_fused(p, n_q) ? indexer_cand_bytes(batch, n_q) : indexer_ws_bytes(batch, n_q, cache_rows);
}

lca_status csa_indexer_topk(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q_idx, const float *w_idx,
                            const lca_bf16 *k_cache, int64_t k_batch_stride, int64_t cache_rows,
                            const int32_t *q_pos, int32_t *out_idx, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
    const char *name = "csa_indexer_topk";
    lca_status st = indexer_validate(name, p, batch, n_q, q_idx, w_idx, k_cache, k_batch_stride, cache_rows, q_pos);
    if (st != LCA_OK) return st;
    LCA_REQUIRE(p->topk >= 1, LCA_ERR_INVALID_ARG, "%s: topk must be positive", name);
    LCA_REQUIRE(out_idx, LCA_ERR_INVALID_ARG, "%s: out_idx is NULL", name);
    const size_t need = csa_indexer_workspace(p, batch, n_q, cache_rows);
    LCA_REQUIRE(workspace && aligned16(workspace) && workspace_bytes >= need, LCA_ERR_WORKSPACE,
                "%s: workspace of %zu bytes (16-byte aligned) needed, got %zu", name, need, workspace_bytes);
    if (indexer_fused(p, n_q)) {
        // prefill: the selection runs in the indexer's epilogue, no score leaves the chip
        IndexerTcArgs a = {};
        a.n_q = n_q;
        a.ratio = p->ratio;
        a.cache_rows = cache_rows;
        a.w = w_idx;
        a.q_pos = q_pos;
        a.k = p->topk;
        a.out_idx = out_idx;
        a.cand = static_cast<uint2 *>(workspace);
        st = indexer_tc_launch<128, 64, 4, true>(batch, n_q, q_idx, k_cache, k_batch_stride, a, stream);
        return st == LCA_OK ? ok() : st;
    }
    const int64_t stride = (cache_rows + 3) & ~(int64_t)3;
    float *scores = static_cast<float *>(workspace);
    st = indexer_launch(p, batch, n_q, q_idx, w_idx, k_cache, k_batch_stride, cache_rows, q_pos, scores, stride,
                        stream);
    if (st != LCA_OK) return st;
    st = topk_launch(p, batch, n_q, scores, stride, q_pos, cache_rows, out_idx, stream);
    return st == LCA_OK ? ok() : st;
}

lca_status csa_indexer_scores_e4m3(const lca_attn_params *p, int batch, int n_q, const uint8_t *q_idx8,
                                   const float *q_scale, const float *w_idx, const uint8_t *k_cache8,
                                   int64_t k_batch_stride, const float *k_scale, int64_t k_scale_batch_stride,
                                   int64_t cache_rows, const int32_t *q_pos, float *scores, int64_t scores_stride,
                                   cudaStream_t stream) {
    const char *name = "csa_indexer_scores_e4m3";
    lca_status st = indexer_e4m3_validate(name, p, batch, n_q, q_idx8, q_scale, w_idx, k_cache8, k_batch_stride,
                                          k_scale, k_scale_batch_stride, cache_rows, q_pos);
    if (st != LCA_OK) return st;
    LCA_REQUIRE(scores && aligned16(scores) && scores_stride >= cache_rows && scores_stride % 4 == 0,
                LCA_ERR_INVALID_ARG, "%s: scores must be 16-byte aligned with a stride >= cache_rows, %% 4", name);
    st = indexer_e4m3_scores_launch(p, batch, n_q, q_idx8, q_scale, w_idx, k_cache8, k_batch_stride, k_scale,
                                    k_scale_batch_stride, cache_rows, q_pos, scores, scores_stride, stream);
    return st == LCA_OK ? ok() : st;
}

lca_status csa_indexer_topk_e4m3(const lca_attn_params *p, int batch, int n_q, const uint8_t *q_idx8,
                                 const float *q_scale, const float *w_idx, const uint8_t *k_cache8,
                                 int64_t k_batch_stride, const float *k_scale, int64_t k_scale_batch_stride,
                                 int64_t cache_rows, const int32_t *q_pos, int32_t *out_idx, void *workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
    const char *name = "csa_indexer_topk_e4m3";
    lca_status st = indexer_e4m3_validate(name, p, batch, n_q, q_idx8, q_scale, w_idx, k_cache8, k_batch_stride,
                                          k_scale, k_scale_batch_stride, cache_rows, q_pos);
    if (st != LCA_OK) return st;
    LCA_REQUIRE(p->topk >= 1, LCA_ERR_INVALID_ARG, "%s: topk must be positive", name);
    LCA_REQUIRE(out_idx, LCA_ERR_INVALID_ARG, "%s: out_idx is NULL", name);
    const size_t need = csa_indexer_workspace(p, batch, n_q, cache_rows);
    LCA_REQUIRE(workspace && aligned16(workspace) && workspace_bytes >= need, LCA_ERR_WORKSPACE,
                "%s: workspace of %zu bytes (16-byte aligned) needed, got %zu", name, need, workspace_bytes);
    if (indexer_fused(p, n_q)) {
        IndexerTcArgs a = indexer_e4m3_args(p, n_q, q_scale, w_idx, k_scale, k_scale_batch_stride, cache_rows, q_pos);
        a.k = p->topk;
        a.out_idx = out_idx;
        a.cand = static_cast<uint2 *>(workspace);
        st = indexer_tc_launch<128, 64, 4, true, true>(batch, n_q, q_idx8, k_cache8, k_batch_stride, a, stream);
        return st == LCA_OK ? ok() : st;
    }
    const int64_t stride = (cache_rows + 3) & ~(int64_t)3;
    float *scores = static_cast<float *>(workspace);
    st = indexer_e4m3_scores_launch(p, batch, n_q, q_idx8, q_scale, w_idx, k_cache8, k_batch_stride, k_scale,
                                    k_scale_batch_stride, cache_rows, q_pos, scores, stride, stream);
    if (st != LCA_OK) return st;
    st = topk_launch(p, batch, n_q, scores, stride, q_pos, cache_rows, out_idx, stream);
    return st == LCA_OK ? ok() : st;
}

size_t csa_attend_workspace(const lca_attn_params *p, int batch, int n_q) {
    if (!p || batch <= 0 || n_q <= 0 || p->topk < 1 || (int64_t)batch * n_q >= kMaxAttendUnits) return 0;
    return plan_attend(p, batch, n_q, (int64_t)p->topk + p->window).total;
}

size_t hca_attend_workspace(const lca_attn_params *p, int batch, int n_q, int64_t cache_rows) {
    if (!p || batch <= 0 || n_q <= 0 || cache_rows <= 0 || (int64_t)batch * n_q >= kMaxAttendUnits) return 0;
    return plan_attend(p, batch, n_q, cache_rows + p->window).total;
}

lca_status csa_attend(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q, const float *gamma_q,
                      const int32_t *q_pos, const lca_bf16 *kv_cache, int64_t kv_batch_stride, int64_t cache_rows,
                      const int32_t *idx, const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                      const float *sink, lca_bf16 *out, float *lse, void *workspace, size_t workspace_bytes,
                      cudaStream_t stream) {
    if (!idx) return fail(LCA_ERR_INVALID_ARG, "csa_attend: idx is NULL");
    return attend_impl("csa_attend", p, batch, n_q, q, gamma_q, q_pos, kv_cache, kv_batch_stride, cache_rows, idx,
                       win_kv, win_batch_stride, win_cap, sink, out, lse, workspace, workspace_bytes, stream);
}

lca_status hca_attend(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q, const float *gamma_q,
                      const int32_t *q_pos, const lca_bf16 *kv_cache, int64_t kv_batch_stride, int64_t cache_rows,
                      const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap, const float *sink,
                      lca_bf16 *out, float *lse, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return attend_impl("hca_attend", p, batch, n_q, q, gamma_q, q_pos, kv_cache, kv_batch_stride, cache_rows, nullptr,
                       win_kv, win_batch_stride, win_cap, sink, out, lse, workspace, workspace_bytes, stream);
}

lca_status csa_attend_e4m3(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q, const float *gamma_q,
                           const int32_t *q_pos, const uint8_t *kv_cache8, int64_t kv_batch_stride,
                           const float *kv_scale, int64_t kv_scale_batch_stride, int64_t cache_rows,
                           const int32_t *idx, const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                           const float *sink, lca_bf16 *out, float *lse, void *workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
    LCA_REQUIRE(idx, LCA_ERR_INVALID_ARG, "csa_attend_e4m3: idx is NULL");
    return attend_impl("csa_attend_e4m3", p, batch, n_q, q, gamma_q, q_pos, nullptr, kv_batch_stride, cache_rows,
                       idx, win_kv, win_batch_stride, win_cap, sink, out, lse, workspace, workspace_bytes, stream,
                       kAttendAll, kv_cache8, kv_scale, kv_scale_batch_stride);
}

lca_status hca_attend_e4m3(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q, const float *gamma_q,
                           const int32_t *q_pos, const uint8_t *kv_cache8, int64_t kv_batch_stride,
                           const float *kv_scale, int64_t kv_scale_batch_stride, int64_t cache_rows,
                           const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap, const float *sink,
                           lca_bf16 *out, float *lse, void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    return attend_impl("hca_attend_e4m3", p, batch, n_q, q, gamma_q, q_pos, nullptr, kv_batch_stride, cache_rows,
                       nullptr, win_kv, win_batch_stride, win_cap, sink, out, lse, workspace, workspace_bytes, stream,
                       kAttendAll, kv_cache8, kv_scale, kv_scale_batch_stride);
}

// ---- hca_attend_noalloc: the dense attention with its scratch in a static device array ----
//
// Some callers cannot hand the library a workspace: a host program with no device allocator
// of its own, or a serving runtime that sizes its device memory once at start-up and may not
// allocate (or free) anything while it serves.  For them the split-K partials and the
// prepared query images live in one file-scope device array, reserved with the module, and
// the entry point makes no allocation of any kind.  The array's address is looked up on
// every call, with the calling thread's current device and context: a context that was torn
// down and created again (cudaDeviceReset, or the primary context released and retained)
// may map the module elsewhere, and a cached address would then point at memory the library
// no longer owns.  The lookup is not a stream operation; on a device's first call it may load
// the module, which is why that first call belongs before any stream capture.  Every call on
// a device shares the one array, so two calls in flight at once on that device (on two
// streams, or from two host threads) overwrite each other's partials; calls must be ordered
// on one stream or otherwise serialised.  No byte of it needs to start at zero: each call
// writes every partial and query image it later reads.
namespace {
constexpr size_t kNoAllocScratchBytes = (size_t)32 << 20;   // 32 MiB
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address in the current context.
static lca_status noalloc_scratch(const char *name, void **addr) {
    void *a = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
    if (e != cudaSuccess || !a) return fail(LCA_ERR_CUDA, "%s: cudaGetSymbolAddress: %s", name, cudaGetErrorString(e));
    *addr = a;
    return LCA_OK;
}

lca_status csa_attend_prepare(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q, const float *gamma_q,
                              const int32_t *q_pos, const lca_bf16 *kv_cache, int64_t kv_batch_stride,
                              int64_t cache_rows, const int32_t *idx, const lca_bf16 *win_kv,
                              int64_t win_batch_stride, int win_cap, const float *sink, lca_bf16 *out, float *lse,
                              void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!idx) return fail(LCA_ERR_INVALID_ARG, "csa_attend_prepare: idx is NULL");
    return attend_impl("csa_attend_prepare", p, batch, n_q, q, gamma_q, q_pos, kv_cache, kv_batch_stride, cache_rows,
                       idx, win_kv, win_batch_stride, win_cap, sink, out, lse, workspace, workspace_bytes, stream,
                       kAttendPrepareOnly);
}

lca_status csa_attend_prepared(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q, const float *gamma_q,
                               const int32_t *q_pos, const lca_bf16 *kv_cache, int64_t kv_batch_stride,
                               int64_t cache_rows, const int32_t *idx, const lca_bf16 *win_kv,
                               int64_t win_batch_stride, int win_cap, const float *sink, lca_bf16 *out, float *lse,
                               void *workspace, size_t workspace_bytes, cudaStream_t stream) {
    if (!idx) return fail(LCA_ERR_INVALID_ARG, "csa_attend_prepared: idx is NULL");
    return attend_impl("csa_attend_prepared", p, batch, n_q, q, gamma_q, q_pos, kv_cache, kv_batch_stride,
                       cache_rows, idx, win_kv, win_batch_stride, win_cap, sink, out, lse, workspace,
                       workspace_bytes, stream, kAttendPrepared);
}

lca_status hca_attend_prepare(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q, const float *gamma_q,
                              const int32_t *q_pos, const lca_bf16 *kv_cache, int64_t kv_batch_stride,
                              int64_t cache_rows, const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                              const float *sink, lca_bf16 *out, float *lse, void *workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
    return attend_impl("hca_attend_prepare", p, batch, n_q, q, gamma_q, q_pos, kv_cache, kv_batch_stride, cache_rows,
                       nullptr, win_kv, win_batch_stride, win_cap, sink, out, lse, workspace, workspace_bytes, stream,
                       kAttendPrepareOnly);
}

lca_status hca_attend_prepared(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q, const float *gamma_q,
                               const int32_t *q_pos, const lca_bf16 *kv_cache, int64_t kv_batch_stride,
                               int64_t cache_rows, const lca_bf16 *win_kv, int64_t win_batch_stride, int win_cap,
                               const float *sink, lca_bf16 *out, float *lse, void *workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
    return attend_impl("hca_attend_prepared", p, batch, n_q, q, gamma_q, q_pos, kv_cache, kv_batch_stride,
                       cache_rows, nullptr, win_kv, win_batch_stride, win_cap, sink, out, lse, workspace,
                       workspace_bytes, stream, kAttendPrepared);
}

extern "C++" {
template <int MT, int KS, int NW>
static void gemv_stream_launch(const GemvStreamArgs &a, int grid, cudaStream_t stream) {
    constexpr int smem = gemv_stream_smem(KS * 256 * NW, MT, NW);
    cudaFuncSetAttribute(gemv_stream_kernel<MT, KS, NW>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    launch_pdl(gemv_stream_kernel<MT, KS, NW>, dim3(grid), dim3(32 * NW), smem, stream, a);
}

// The streaming product's variants: 8 warps (16 measured slower), K / 2048 slices of 256 per
// warp, M x K / 2048 <= 16 activations per lane.  Returns false for shapes it does not cover.
template <int MT>
static bool gemv_stream_dispatch_mt(const GemvStreamArgs &a, int grid, cudaStream_t stream) {
    switch (a.K) {
    case 2048: gemv_stream_launch<MT, 1, 8>(a, grid, stream); return true;
    case 4096: gemv_stream_launch<MT, 2, 8>(a, grid, stream); return true;
    case 6144: if constexpr (MT <= 4) { gemv_stream_launch<MT, 3, 8>(a, grid, stream); return true; } return false;
    case 8192: if constexpr (MT <= 4) { gemv_stream_launch<MT, 4, 8>(a, grid, stream); return true; } return false;
    default: return false;
    }
}

static bool gemv_stream_dispatch(const GemvStreamArgs &a, int mt, int grid, cudaStream_t stream) {
    switch (mt) {
    case 1: return gemv_stream_dispatch_mt<1>(a, grid, stream);
    case 2: return gemv_stream_dispatch_mt<2>(a, grid, stream);
    case 4: return gemv_stream_dispatch_mt<4>(a, grid, stream);
    case 8: return gemv_stream_dispatch_mt<8>(a, grid, stream);
    default: return false;
    }
}
}  // extern "C++"

// C = A . B^T for the batches' weight blocks.  The streaming kernel takes weight arrays stored
// contiguously ([batches][N][K]) with K one of 2048, 4096, 6144, 8192, N a multiple of 4 and
// few enough activations per lane (gemv_stream_dispatch); everything else takes gemv_kernel.
// b_early: the weights may be read before the previous kernel in the stream has finished.
static lca_status gemv_launch(const char *name, int M, int N, int K, const lca_bf16 *A, int64_t lda, int64_t a_off,
                              const lca_bf16 *B, int64_t ldb, int64_t b_off, lca_bf16 *C, int64_t ldc, int64_t c_off,
                              int batches, cudaStream_t stream, bool b_early = false) {
    const int mt = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16;
    if ((K == 2048 || K == 4096 || K == 6144 || K == 8192) && mt <= 8 && ldb == K &&
        (batches == 1 || b_off == (int64_t)N * K) && N % 4 == 0 && aligned16(A) && aligned16(B) && lda % 8 == 0 &&
        a_off % 8 == 0) {
        GemvStreamArgs g;
        g.M = M;
        g.N = N;
        g.K = K;
        g.groups = (int64_t)batches * N / kGsRows;
        g.A = reinterpret_cast<const __nv_bfloat16 *>(A);
        g.lda = lda;
        g.a_batch_off = a_off;
        g.B = reinterpret_cast<const __nv_bfloat16 *>(B);
        g.C = reinterpret_cast<__nv_bfloat16 *>(C);
        g.ldc = ldc;
        g.c_batch_off = c_off;
        g.b_early = b_early ? 1 : 0;
        const int grid = (int)std::min<int64_t>(g.groups, device_sm_count());
        if (gemv_stream_dispatch(g, mt, grid, stream)) return check_launch(name);
    }
    GemvArgs a;
    a.M = M;
    a.N = N;
    a.K = K;
    a.A = reinterpret_cast<const __nv_bfloat16 *>(A);
    a.lda = lda;
    a.a_batch_off = a_off;
    a.B = reinterpret_cast<const __nv_bfloat16 *>(B);
    a.ldb = ldb;
    a.b_batch_off = b_off;
    a.C = reinterpret_cast<__nv_bfloat16 *>(C);
    a.ldc = ldc;
    a.c_batch_off = c_off;
    const int rows_per_block = (kGemvThreads / 32) * kGemvRowsPerWarp;
    dim3 grid((unsigned)ceil_div64(N, rows_per_block), batches);
    if (M <= 1) launch_pdl(gemv_kernel<1>, grid, dim3(kGemvThreads), 0, stream, a);
    else if (M <= 2) launch_pdl(gemv_kernel<2>, grid, dim3(kGemvThreads), 0, stream, a);
    else if (M <= 4) launch_pdl(gemv_kernel<4>, grid, dim3(kGemvThreads), 0, stream, a);
    else if (M <= 8) launch_pdl(gemv_kernel<8>, grid, dim3(kGemvThreads), 0, stream, a);
    else launch_pdl(gemv_kernel<16>, grid, dim3(kGemvThreads), 0, stream, a);
    return check_launch(name);
}

lca_status hca_attend_noalloc(const lca_attn_params *p, int batch, int n_q, const lca_bf16 *q,
                              const float *gamma_q, const int32_t *q_pos, const lca_bf16 *kv_cache,
                              int64_t kv_batch_stride, int64_t cache_rows, const lca_bf16 *win_kv,
                              int64_t win_batch_stride, int win_cap, const float *sink, lca_bf16 *out, float *lse,
                              cudaStream_t stream) {
    const char *name = "hca_attend_noalloc";
    lca_status st = attend_validate(name, p, batch, n_q);
    if (st != LCA_OK) return st;
    LCA_REQUIRE(cache_rows > 0, LCA_ERR_INVALID_ARG, "%s: cache_rows must be positive", name);
    const size_t need = plan_attend(p, batch, n_q, cache_rows + p->window).total;
    LCA_REQUIRE(need <= kNoAllocScratchBytes, LCA_ERR_WORKSPACE,
                "%s: this call needs %zu bytes of scratch, more than the %zu-byte static array "
                "(use hca_attend with a workspace)", name, need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    st = noalloc_scratch(name, &scratch);
    if (st != LCA_OK) return st;
    return attend_impl(name, p, batch, n_q, q, gamma_q, q_pos, kv_cache, kv_batch_stride, cache_rows, nullptr, win_kv,
                       win_batch_stride, win_cap, sink, out, lse, scratch, kNoAllocScratchBytes, stream);
}

// The tensor-core product: 128-row tiles of C, BN = 64, 128 or 256 columns by N.
static lca_status gemm_tc_launch(const char *name, int M, int N, int K, const lca_bf16 *A, int64_t lda,
                                 const lca_bf16 *B, int64_t ldb, void *C, int64_t ldc, bool f32_out,
                                 cudaStream_t stream) {
    const int BN = N <= 64 ? 64 : N <= 128 ? 128 : 256;
    CUtensorMap a_map, b_map;
    const uint64_t ad[2] = {(uint64_t)K, (uint64_t)M}, bd[2] = {(uint64_t)K, (uint64_t)N};
    const uint64_t as[1] = {(uint64_t)lda * 2}, bs[1] = {(uint64_t)ldb * 2};
    const uint32_t abox[2] = {(uint32_t)kGtBK, (uint32_t)kGtBM}, bbox[2] = {(uint32_t)kGtBK, (uint32_t)BN};
    if (!make_tensor_map(&a_map, A, 2, ad, as, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&b_map, B, 2, bd, bs, bbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return fail(LCA_ERR_CUDA, "%s: tensor map rejected by the driver", name);
    GemmTcArgs g;
    g.M = M;
    g.N = N;
    g.K = K;
    g.C = C;
    g.ldc = ldc;
    const dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + kGtBM - 1) / kGtBM));
#define LCA_GEMM_TC(BNV, F32)                                                                                      \
    do {                                                                                                           \
        cudaFuncSetAttribute(gemm_tc_kernel<BNV, F32>, cudaFuncAttributeMaxDynamicSharedMemorySize,                \
                             GemmTcConfig<BNV>::SMEM_BYTES);                                                       \
        launch_pdl(gemm_tc_kernel<BNV, F32>, grid, dim3(kGtThreads), GemmTcConfig<BNV>::SMEM_BYTES, stream, a_map, \
                   b_map, g);                                                                                      \
    } while (0)
    if (f32_out) {
        if (BN == 64) LCA_GEMM_TC(64, true);
        else if (BN == 128) LCA_GEMM_TC(128, true);
        else LCA_GEMM_TC(256, true);
    } else {
        if (BN == 64) LCA_GEMM_TC(64, false);
        else if (BN == 128) LCA_GEMM_TC(128, false);
        else LCA_GEMM_TC(256, false);
    }
#undef LCA_GEMM_TC
    return check_launch(name);
}

static lca_status gemm_validate(const char *name, int M, int N, int K, const void *A, int64_t lda, const void *B,
                                int64_t ldb, const void *C, int64_t ldc) {
    LCA_REQUIRE(M >= 1 && N >= 1 && K >= 8 && K % 8 == 0, LCA_ERR_UNSUPPORTED,
                "%s: need M, N >= 1 and K a positive multiple of 8 (M=%d N=%d K=%d)", name, M, N, K);
    LCA_REQUIRE(A && B && C, LCA_ERR_INVALID_ARG, "%s: a required pointer is NULL", name);
    LCA_REQUIRE(aligned16(A) && aligned16(B) && lda % 8 == 0 && ldb % 8 == 0 && lda >= K && ldb >= K && ldc >= N,
                LCA_ERR_INVALID_ARG, "%s: A and B must be 16-byte aligned with strides >= K, multiples of 8", name);
    return LCA_OK;
}

lca_status lca_gemm_bf16(int M, int N, int K, const lca_bf16 *A, int64_t lda, const lca_bf16 *B, int64_t ldb,
                         lca_bf16 *C, int64_t ldc, cudaStream_t stream) {
    const char *name = "lca_gemm_bf16";
    lca_status st = gemm_validate(name, M, N, K, A, lda, B, ldb, C, ldc);
    if (st != LCA_OK) return st;
    if (M <= 16) {
        st = gemv_launch(name, M, N, K, A, lda, 0, B, ldb, 0, C, ldc, 0, 1, stream);
    } else {
        st = gemm_tc_launch(name, M, N, K, A, lda, B, ldb, C, ldc, false, stream);
    }
    return st == LCA_OK ? ok() : st;
}

lca_status lca_gemm_bf16_f32(int M, int N, int K, const lca_bf16 *A, int64_t lda, const lca_bf16 *B, int64_t ldb,
                             float *C, int64_t ldc, cudaStream_t stream) {
    const char *name = "lca_gemm_bf16_f32";
    lca_status st = gemm_validate(name, M, N, K, A, lda, B, ldb, C, ldc);
    if (st != LCA_OK) return st;
    st = gemm_tc_launch(name, M, N, K, A, lda, B, ldb, C, ldc, true, stream);
    return st == LCA_OK ? ok() : st;
}

// ---- manifold-constrained hyper-connections ----
static lca_status mhc_validate(const char *name, int T, int n, int d) {
    LCA_REQUIRE(T >= 1, LCA_ERR_INVALID_ARG, "%s: T must be positive", name);
    LCA_REQUIRE(n == 1 || n == 2 || n == 4, LCA_ERR_UNSUPPORTED, "%s: n = %d streams not in {1, 2, 4}", name, n);
    LCA_REQUIRE(d >= 8 && d % 8 == 0 && d <= 65536, LCA_ERR_UNSUPPORTED,
                "%s: d = %d must be a multiple of 8 in [8, 65536]", name, d);
    return LCA_OK;
}

size_t lca_mhc_workspace(int T, int n) {
    (void)T;
    (void)n;
    return 0;   // the generated values stay in the product's tensor memory
}

lca_status lca_mhc_pre(int T, int n, int d, int iters, const lca_bf16 *x, const lca_bf16 *phi, const float *bias,
                       lca_bf16 *h, float *a, float *c, float *b_mix, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream) {
    const char *name = "lca_mhc_pre";
    (void)workspace;
    (void)workspace_bytes;
    lca_status st = mhc_validate(name, T, n, d);
    if (st != LCA_OK) return st;
    LCA_REQUIRE(iters >= 1 && iters <= 1000, LCA_ERR_INVALID_ARG, "%s: iters = %d not in [1, 1000]", name, iters);
    LCA_REQUIRE(x && phi && bias && h && a && c && b_mix, LCA_ERR_INVALID_ARG, "%s: a required pointer is NULL", name);
    LCA_REQUIRE(aligned16(x) && aligned16(phi) && aligned16(h), LCA_ERR_INVALID_ARG,
                "%s: x, phi and h must be 16-byte aligned", name);
    // the generated values and, in the product's epilogue, the coefficients
    const int K = 2 * n + n * n, nd = n * d;
    CUtensorMap a_map, b_map;
    const uint64_t ad[2] = {(uint64_t)nd, (uint64_t)T}, bd[2] = {(uint64_t)nd, (uint64_t)K};
    const uint64_t st_row[1] = {(uint64_t)nd * 2};
    const uint32_t abox[2] = {(uint32_t)kGtBK, (uint32_t)kGtBM}, bbox[2] = {(uint32_t)kGtBK, 64u};
    if (!make_tensor_map(&a_map, x, 2, ad, st_row, abox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tensor_map(&b_map, phi, 2, bd, st_row, bbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return fail(LCA_ERR_CUDA, "%s: tensor map rejected by the driver", name);
    GemmTcArgs g = {};
    g.M = T;
    g.N = K;
    g.K = nd;
    g.mhc.bias = bias;
    g.mhc.a = a;
    g.mhc.c = c;
    g.mhc.B = b_mix;
    g.mhc.iters = iters;
    const dim3 grid(1, (unsigned)((T + kGtBM - 1) / kGtBM));
    constexpr int smem = GemmTcConfig<64>::SMEM_BYTES;
    switch (n) {
    case 1:
        cudaFuncSetAttribute(gemm_tc_kernel<64, true, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        launch_pdl(gemm_tc_kernel<64, true, 1>, grid, dim3(kGtThreads), smem, stream, a_map, b_map, g);
        break;
    case 2:
        cudaFuncSetAttribute(gemm_tc_kernel<64, true, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        launch_pdl(gemm_tc_kernel<64, true, 2>, grid, dim3(kGtThreads), smem, stream, a_map, b_map, g);
        break;
    default:
        cudaFuncSetAttribute(gemm_tc_kernel<64, true, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        launch_pdl(gemm_tc_kernel<64, true, 4>, grid, dim3(kGtThreads), smem, stream, a_map, b_map, g);
        break;
    }
    st = check_launch(name);
    if (st != LCA_OK) return st;
    MhcMixArgs m = {};
    m.d = d;
    m.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    m.a = a;
    m.h = reinterpret_cast<__nv_bfloat16 *>(h);
    const dim3 mgrid((unsigned)ceil_div64(d / 8, kMhcThreads), (unsigned)T);
    switch (n) {
    case 1: launch_pdl(mhc_pre_mix_kernel<1>, mgrid, dim3(kMhcThreads), 0, stream, m); break;
    case 2: launch_pdl(mhc_pre_mix_kernel<2>, mgrid, dim3(kMhcThreads), 0, stream, m); break;
    default: launch_pdl(mhc_pre_mix_kernel<4>, mgrid, dim3(kMhcThreads), 0, stream, m); break;
    }
    st = check_launch(name);
    return st == LCA_OK ? ok() : st;
}

lca_status lca_mhc_post(int T, int n, int d, const lca_bf16 *x, const float *b_mix, const float *c, const lca_bf16 *y,
                        lca_bf16 *x_out, cudaStream_t stream) {
    const char *name = "lca_mhc_post";
    lca_status st = mhc_validate(name, T, n, d);
    if (st != LCA_OK) return st;
    LCA_REQUIRE(x && b_mix && c && y && x_out, LCA_ERR_INVALID_ARG, "%s: a required pointer is NULL", name);
    LCA_REQUIRE(aligned16(x) && aligned16(y) && aligned16(x_out), LCA_ERR_INVALID_ARG,
                "%s: x, y and x_out must be 16-byte aligned", name);
    MhcMixArgs m = {};
    m.d = d;
    m.x = reinterpret_cast<const __nv_bfloat16 *>(x);
    m.B = b_mix;
    m.c = c;
    m.y = reinterpret_cast<const __nv_bfloat16 *>(y);
    m.x_out = reinterpret_cast<__nv_bfloat16 *>(x_out);
    const dim3 mgrid((unsigned)ceil_div64(d / 8, kMhcThreads), (unsigned)T);
    switch (n) {
    case 1: launch_pdl(mhc_post_kernel<1>, mgrid, dim3(kMhcThreads), 0, stream, m); break;
    case 2: launch_pdl(mhc_post_kernel<2>, mgrid, dim3(kMhcThreads), 0, stream, m); break;
    default: launch_pdl(mhc_post_kernel<4>, mgrid, dim3(kMhcThreads), 0, stream, m); break;
    }
    st = check_launch(name);
    return st == LCA_OK ? ok() : st;
}

lca_status lca_grouped_oproj(int batch, int heads, int head_dim, int groups, int d_g, int d_model, const lca_bf16 *o,
                             const lca_bf16 *Wg, const lca_bf16 *Wm, lca_bf16 *mid, lca_bf16 *y,
                             cudaStream_t stream) {
    const char *name = "lca_grouped_oproj";
    LCA_REQUIRE(batch >= 1 && batch <= 16, LCA_ERR_UNSUPPORTED, "%s: batch %d not in [1, 16]", name, batch);
    LCA_REQUIRE(heads >= 1 && groups >= 1 && heads % groups == 0 && head_dim >= 1 && d_g >= 1 && d_model >= 1,
                LCA_ERR_INVALID_ARG, "%s: heads must divide into groups", name);
    const int64_t in_g = (int64_t)(heads / groups) * head_dim;
    LCA_REQUIRE(in_g % 8 == 0 && ((int64_t)groups * d_g) % 8 == 0 && d_g % 8 == 0, LCA_ERR_UNSUPPORTED,
                "%s: group input and output widths must be multiples of 8", name);
    LCA_REQUIRE(o && Wg && Wm && mid && y, LCA_ERR_INVALID_ARG, "%s: a required pointer is NULL", name);
    LCA_REQUIRE(aligned16(o) && aligned16(Wg) && aligned16(Wm) && aligned16(mid), LCA_ERR_INVALID_ARG,
                "%s: o, Wg, Wm and mid must be 16-byte aligned", name);
    const int64_t hc = (int64_t)heads * head_dim;
    const int64_t gd = (int64_t)groups * d_g;
    lca_status st = gemv_launch(name, batch, d_g, (int)in_g, o, hc, in_g, Wg, in_g, (int64_t)d_g * in_g, mid, gd, d_g,
                                groups, stream, true);
    if (st != LCA_OK) return st;
    st = gemv_launch(name, batch, d_model, (int)gd, mid, gd, 0, Wm, gd, 0, y, d_model, 0, 1, stream, true);
    return st == LCA_OK ? ok() : st;
}

}  // extern "C"

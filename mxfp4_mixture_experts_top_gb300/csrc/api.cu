// Host side of the C ABI: argument validation, tensor-map encoding and
// caching, workspace layout, launches. Every entry point enqueues on the
// caller's stream only and returns before the device work finishes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/moe_mxfp4.h"
#include "moe_internal.h"
#include "mxfp4_tile.cuh"

namespace moe {

static std::atomic<unsigned long long> g_launches{0};
void note_launch(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

struct MapKey {
    int dev, kind;
    const void *ptr;
    uint64_t d0, d1, d2;
    uint32_t b1, b3;
    bool operator<(const MapKey &o) const
    {
        return std::tie(dev, kind, ptr, d0, d1, d2, b1, b3) < std::tie(o.dev, o.kind, o.ptr, o.d0, o.d1, o.d2, o.b1, o.b3);
    }
};

struct MapEntry {
    CUtensorMap map;
};

std::mutex g_map_mu;
std::map<MapKey, MapEntry> g_maps;

// Cached tensor map. kind 0: prepacked weight nibbles, a 2-D tensor of d1 rows of 128 E2M1 values
// (64 B) read as "16 x U4, 16-byte aligned" (each 8-byte group lands in 16 bytes of shared memory),
// box 128 x b1 rows. kind 1: activation terms, a 4-D uint8 tensor [d0 / 128 slabs][d2 terms]
// [d1 rows][128], box 128 x b1 rows x d2 terms x b3 slabs. Both with the 128-byte swizzle of the
// MMA operands. kind 2: activation scale words, a 3-D uint32 tensor [d2 slabs][d1 terms][d0 rows],
// box b1 rows x d1 terms x b3 slabs, no swizzle.
// The map is copied out under the cache lock, so a later eviction (the cache is emptied once it
// holds 4096 maps) or another thread cannot invalidate what the caller holds.
bool get_map(CUtensorMap *out, int kind, const void *ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b1,
             uint32_t b3, moe_status_t *st)
{
    int dev = 0;
    cudaGetDevice(&dev);
    MapKey key{dev, kind, ptr, d0, d1, d2, b1, b3};
    std::lock_guard<std::mutex> lk(g_map_mu);
    auto it = g_maps.find(key);
    if (it != g_maps.end()) {
        *out = it->second.map;
        return true;
    }
    EncodeTiledFn fn = encode_fn();
    if (!fn) { *st = MOE_ERR_CUDA; return false; }
    if (g_maps.size() > 4096) g_maps.clear();
    MapEntry ent;
    CUresult r;
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (kind == 0) {
        cuuint64_t dims[2] = {128, d1};
        cuuint64_t strides[1] = {64};
        cuuint32_t box[2] = {128, b1};
        r = fn(&ent.map, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else if (kind == 1) {
        cuuint64_t dims[4] = {128, d1, d2, d0 / 128};
        cuuint64_t strides[3] = {128, 128 * d1, 128 * d1 * d2};
        cuuint32_t box[4] = {128, b1, (cuuint32_t)d2, b3};
        r = fn(&ent.map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        cuuint64_t dims[3] = {d0, d1, d2};
        cuuint64_t strides[2] = {d0 * 4, d0 * d1 * 4};
        cuuint32_t box[3] = {b1, (cuuint32_t)d1, b3};
        r = fn(&ent.map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    if (r != CUDA_SUCCESS) { *st = MOE_ERR_CUDA; return false; }
    g_maps.emplace(key, ent);
    *out = ent.map;
    return true;
}

int sm_count()
{
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    return n;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

moe_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status_t check_desc(const moe_layer_desc *d)
{
    if (!d) return MOE_ERR_INVALID_ARG;
    if (d->T < 0 || d->H <= 0 || d->I <= 0 || d->E <= 0 || d->k <= 0 || d->k > d->E) return MOE_ERR_INVALID_ARG;
    if (d->flags & ~MOE_FLAG_FAST_COMBINE) return MOE_ERR_INVALID_ARG;
    if (d->out_dtype != MOE_OUT_F32 && d->out_dtype != MOE_OUT_BF16) return MOE_ERR_INVALID_ARG;
    if (d->E > 1024 || d->k > 32) return MOE_ERR_UNSUPPORTED;
    if (d->H % 128 || d->I % 128) return MOE_ERR_UNSUPPORTED;
    if (d->block_m != 16 && d->block_m != 32 && d->block_m != 64 && d->block_m != 128) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)d->T * d->k > (int64_t)INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Layout {
    size_t err, xq, xs, hq, hs, staging, total;
};

// Rows of the activation scale-word arrays: the permutation rows rounded up to 4 (TMA strides are
// multiples of 16 bytes).
int64_t scale_rows(const moe_layer_desc *d)
{
    return (moe_permute_rows_capacity(d->T, d->E, d->k, d->block_m) + 3) / 4 * 4;
}

Layout workspace_layout(const moe_layer_desc *d)
{
    const int NT_H = regime_nt_h(pick_regime(d->T, d->k, d->E, d->H));
    const int64_t P = (int64_t)d->T * d->k;
    const int64_t R = moe_permute_rows_capacity(d->T, d->E, d->k, d->block_m);
    const int64_t RS = scale_rows(d);
    Layout L;
    L.err = 0;
    L.xq = 4096;                 // error word at 0, fused-decode expert counters from byte 256
    L.xs = align_up(L.xq + (size_t)NT_X * R * d->H, 1024);
    L.hq = align_up(L.xs + (size_t)NT_X * RS * (d->H / 32), 1024);
    L.hs = align_up(L.hq + (size_t)NT_H * R * d->I, 1024);
    L.staging = align_up(L.hs + (size_t)NT_H * RS * (d->I / 32), 1024);
    L.total = align_up(L.staging + (size_t)P * d->H * 4, 1024);
    return L;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return MOE_ABI_VERSION; }

const char *moe_status_string(moe_status_t s)
{
    switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_MISALIGNED: return "pointer not 16-byte aligned (the forward workspace: 256-byte)";
    case MOE_ERR_WORKSPACE: return "workspace or packed buffer too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE: return "device-detected invalid input (expert id out of range)";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

uint64_t moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status_t moe_route(const float *d_logits, int T, int E, int k, int32_t *d_topk_ids, float *d_topk_w,
                       uint32_t *d_bitmatrix, void *stream)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!d_logits || !d_topk_ids || !d_topk_w) return MOE_ERR_INVALID_ARG;
    if (!aligned16(d_logits) || !aligned16(d_topk_ids) || !aligned16(d_topk_w) ||
        (d_bitmatrix && !aligned16(d_bitmatrix)))
        return MOE_ERR_MISALIGNED;
    return from_cuda(launch_route(d_logits, T, E, k, d_topk_ids, d_topk_w, d_bitmatrix, (cudaStream_t)stream));
}

size_t moe_permute_workspace_size(int T, int E, int k, int block_m)
{
    (void)T;
    (void)E;
    (void)k;
    (void)block_m;
    return 0;   // the permutation keeps its scratch (histograms, scans) in shared memory
}

void moe_clear_cache(void)
{
    std::lock_guard<std::mutex> lk(g_map_mu);
    g_maps.clear();
}

int64_t moe_permute_rows_capacity(int T, int E, int k, int block_m)
{
    if (T < 0 || E <= 0 || k <= 0 || block_m <= 0) return 0;
    const int64_t P = (int64_t)T * k;
    const int64_t used = P < E ? P : E;
    return P + used * (block_m - 1);
}

moe_status_t moe_permute(const int32_t *d_topk_ids, int T, int E, int k, int block_m, int32_t *d_counts,
                         int32_t *d_offsets, int32_t *d_padded_offsets, int32_t *d_row_to_pair,
                         int32_t *d_pair_to_row, int32_t *d_error, void *stream)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED;
    if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)T * k > (int64_t)INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if (!d_counts || !d_offsets || !d_padded_offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!d_topk_ids || !d_row_to_pair || !d_pair_to_row)) return MOE_ERR_INVALID_ARG;
    const void *ptrs[] = {d_topk_ids, d_counts, d_offsets, d_padded_offsets, d_row_to_pair, d_pair_to_row, d_error};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return MOE_ERR_MISALIGNED;
    const int64_t cap = moe_permute_rows_capacity(T, E, k, block_m);
    return from_cuda(launch_permute(d_topk_ids, T, E, k, block_m, d_counts, d_offsets, d_padded_offsets,
                                    d_row_to_pair, cap, d_pair_to_row, d_error, (cudaStream_t)stream));
}

moe_status_t moe_route_permute(const float *d_logits, int T, int E, int k, int block_m, int32_t *d_topk_ids,
                               float *d_topk_w, uint32_t *d_bitmatrix, int32_t *d_counts, int32_t *d_offsets,
                               int32_t *d_padded_offsets, int32_t *d_row_to_pair, int32_t *d_pair_to_row,
                               int32_t *d_error, void *stream)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED;
    if (block_m != 16 && block_m != 32 && block_m != 64 && block_m != 128) return MOE_ERR_UNSUPPORTED;
    if ((int64_t)T * k > (int64_t)INT32_MAX / 2) return MOE_ERR_UNSUPPORTED;
    if (!d_counts || !d_offsets || !d_padded_offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!d_logits || !d_topk_ids || !d_topk_w || !d_row_to_pair || !d_pair_to_row)) return MOE_ERR_INVALID_ARG;
    const void *ptrs[] = {d_logits, d_topk_ids, d_topk_w, d_bitmatrix, d_counts, d_offsets, d_padded_offsets,
                          d_row_to_pair, d_pair_to_row, d_error};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return MOE_ERR_MISALIGNED;
    const int64_t cap = moe_permute_rows_capacity(T, E, k, block_m);
    return from_cuda(launch_route_permute(d_logits, T, E, k, block_m, d_topk_ids, d_topk_w, d_bitmatrix, d_counts,
                                          d_offsets, d_padded_offsets, d_row_to_pair, cap, d_pair_to_row, d_error,
                                          (cudaStream_t)stream));
}

size_t moe_mxfp4_packed_bytes(const moe_layer_desc *d)
{
    if (!d || d->E <= 0 || d->H <= 0 || d->I <= 0 || d->H % 128 || d->I % 128) return 0;
    return packed_w13_bytes(d->E, d->H, d->I) + packed_w2_bytes(d->E, d->H, d->I);
}

moe_status_t moe_mxfp4_prepack(const moe_layer_desc *d, const uint8_t *d_w13_q, const uint8_t *d_w13_s,
                               const uint8_t *d_w2_q, const uint8_t *d_w2_s, void *d_packed, size_t packed_bytes,
                               void *stream)
{
    moe_status_t st = check_desc(d);
    if (st != MOE_OK) return st;
    if (!d_w13_q || !d_w13_s || !d_w2_q || !d_w2_s || !d_packed) return MOE_ERR_INVALID_ARG;
    if (!aligned16(d_w13_q) || !aligned16(d_w13_s) || !aligned16(d_w2_q) || !aligned16(d_w2_s) ||
        !aligned16(d_packed))
        return MOE_ERR_MISALIGNED;
    if (packed_bytes < moe_mxfp4_packed_bytes(d)) return MOE_ERR_WORKSPACE;
    return from_cuda(launch_prepack(d_w13_q, d_w13_s, d_w2_q, d_w2_s, d->E, d->H, d->I,
                                    static_cast<uint8_t *>(d_packed), (cudaStream_t)stream));
}

moe_status_t moe_mxfp4_dequant_bf16(const moe_layer_desc *d, const void *d_packed, int which, int expert,
                                    uint16_t *d_out, void *stream)
{
    moe_status_t st = check_desc(d);
    if (st != MOE_OK) return st;
    if (!d_packed || !d_out || (which != 0 && which != 1) || expert < 0 || expert >= d->E)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(d_packed) || !aligned16(d_out)) return MOE_ERR_MISALIGNED;
    return from_cuda(launch_dequant(static_cast<const uint8_t *>(d_packed), which, expert, d->E, d->H, d->I, d_out,
                                    (cudaStream_t)stream));
}

size_t moe_mxfp4_workspace_bytes(const moe_layer_desc *d)
{
    if (check_desc(d) != MOE_OK) return 0;
    return workspace_layout(d).total;
}

moe_status_t moe_mxfp4_workspace_layout(const moe_layer_desc *d, size_t out[7])
{
    moe_status_t st = check_desc(d);
    if (st != MOE_OK) return st;
    if (!out) return MOE_ERR_INVALID_ARG;
    Layout L = workspace_layout(d);
    out[0] = L.err;
    out[1] = L.xq;
    out[2] = L.xs;
    out[3] = L.hq;
    out[4] = L.hs;
    out[5] = L.staging;
    out[6] = L.total;
    return MOE_OK;
}

moe_status_t moe_mxfp4_forward_plan(const moe_layer_desc *d, int out[4])
{
    moe_status_t st = check_desc(d);
    if (st != MOE_OK) return st;
    if (!out) return MOE_ERR_INVALID_ARG;
    const Regime rg = pick_regime(d->T, d->k, d->E, d->H);
    const ForwardPlan pl = plan_forward(rg, d->H, d->I, d->E, (d->flags & MOE_FLAG_FAST_COMBINE) != 0,
                                        d->out_dtype == MOE_OUT_BF16, false);
    out[0] = (int)rg;
    out[1] = pl.fused ? 1 : 0;
    out[2] = pl.fast ? 1 : 0;
    out[3] = pl.launches;
    return MOE_OK;
}

moe_status_t moe_mxfp4_forward_timed(const moe_layer_desc *d, const uint16_t *d_x, const void *d_packed,
                                     const float *d_topk_w, const int32_t *d_offsets,
                                     const int32_t *d_padded_offsets, const int32_t *d_row_to_pair, void *d_y,
                                     void *d_workspace, size_t workspace_bytes, void *const *events, void *stream)
{
    moe_status_t st = check_desc(d);
    if (st != MOE_OK) return st;
    if (d->T == 0) return MOE_OK;
    const void *ptrs[] = {d_x, d_packed, d_topk_w, d_offsets, d_padded_offsets, d_row_to_pair, d_y, d_workspace};
    for (const void *p : ptrs)
        if (!p) return MOE_ERR_INVALID_ARG;
    for (const void *p : ptrs)
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    if (reinterpret_cast<uintptr_t>(d_workspace) & 255u) return MOE_ERR_MISALIGNED;   // 32-byte stores inside
    Layout L = workspace_layout(d);
    if (workspace_bytes < L.total) return MOE_ERR_WORKSPACE;
    cudaStream_t s = (cudaStream_t)stream;
    uint8_t *ws = static_cast<uint8_t *>(d_workspace);
    const int64_t R = moe_permute_rows_capacity(d->T, d->E, d->k, d->block_m);

    ForwardArgs a{};
    a.T = d->T;
    a.H = d->H;
    a.I = d->I;
    a.E = d->E;
    a.k = d->k;
    a.block_m = d->block_m;
    a.swiglu_limit = d->swiglu_limit;
    a.fast_combine = (d->flags & MOE_FLAG_FAST_COMBINE) != 0;   // launch_forward decides where it applies
    a.rows_cap = R;
    a.rows_sf = scale_rows(d);
    a.x = d_x;
    a.packed = static_cast<const uint8_t *>(d_packed);
    a.topk_w = d_topk_w;
    a.offsets = d_offsets;
    a.padded = d_padded_offsets;
    a.row_to_pair = d_row_to_pair;
    a.y = d_y;
    a.done13 = reinterpret_cast<uint32_t *>(ws + L.err + 256);
    a.y_bf16 = d->out_dtype == MOE_OUT_BF16;
    a.dev_error = reinterpret_cast<int32_t *>(ws + L.err);
    a.xq = ws + L.xq;
    a.xs = ws + L.xs;
    a.hq = ws + L.hq;
    a.hs = ws + L.hs;
    a.staging = reinterpret_cast<float *>(ws + L.staging);
    a.num_sms = sm_count();
    a.events = events;
    a.regime = pick_regime(d->T, d->k, d->E, d->H);
    const uint32_t sps = (uint32_t)regime_sps(a.regime);
    const uint8_t *w13 = a.packed, *w2 = a.packed + packed_w13_bytes(d->E, d->H, d->I);
    const uint64_t rows13 = (uint64_t)d->E * 2 * d->I * (d->H / KSLAB);   // 128-element rows of W13 nibbles
    const uint64_t rows2 = (uint64_t)d->E * d->H * (d->I / KSLAB);
    if (!get_map(&a.tmap_w13, 0, w13, 128, rows13, 1, 128 * sps, 1, &st)) return st;
    if (!get_map(&a.tmap_w13_1, 0, w13, 128, rows13, 1, 128, 1, &st)) return st;
    if (!get_map(&a.tmap_w2, 0, w2, 128, rows2, 1, 128 * sps, 1, &st)) return st;
    if (!get_map(&a.tmap_w2_1, 0, w2, 128, rows2, 1, 128, 1, &st)) return st;
    const uint32_t n13 = (uint32_t)regime_nmax(a.regime, 0), n2 = (uint32_t)regime_nmax(a.regime, 1);
    const uint64_t NT_H = (uint64_t)regime_nt_h(a.regime);
    const uint64_t s13 = (uint64_t)(d->H / KSLAB), s2 = (uint64_t)(d->I / KSLAB);
    // activation terms and their scale words: a whole stage (sps slabs) per box, and single-slab
    // boxes for a stage that straddles two tiles
    if (!get_map(&a.tmap_xq, 1, a.xq, (uint64_t)d->H, (uint64_t)R, NT_X, n13, sps, &st)) return st;
    if (!get_map(&a.tmap_xq1, 1, a.xq, (uint64_t)d->H, (uint64_t)R, NT_X, n13, 1, &st)) return st;
    if (!get_map(&a.tmap_hq, 1, a.hq, (uint64_t)d->I, (uint64_t)R, NT_H, n2, sps, &st)) return st;
    if (!get_map(&a.tmap_hq1, 1, a.hq, (uint64_t)d->I, (uint64_t)R, NT_H, n2, 1, &st)) return st;
    if (!get_map(&a.tmap_xs, 2, a.xs, (uint64_t)a.rows_sf, NT_X, s13, n13, sps, &st)) return st;
    if (!get_map(&a.tmap_xs1, 2, a.xs, (uint64_t)a.rows_sf, NT_X, s13, n13, 1, &st)) return st;
    if (!get_map(&a.tmap_hs, 2, a.hs, (uint64_t)a.rows_sf, NT_H, s2, n2, sps, &st)) return st;
    if (!get_map(&a.tmap_hs1, 2, a.hs, (uint64_t)a.rows_sf, NT_H, s2, n2, 1, &st)) return st;
    // at most 8 tokens: no expert holds more than 8 rows, and the fused decode GEMMs take 8-row tiles
    a.rows8 = d->T <= 8 && a.regime == Regime::Tiny;
    if (a.rows8) {
        if (!get_map(&a.tmap_xq8, 1, a.xq, (uint64_t)d->H, (uint64_t)R, NT_X, 8, sps, &st)) return st;
        if (!get_map(&a.tmap_hq8, 1, a.hq, (uint64_t)d->I, (uint64_t)R, NT_H, 8, sps, &st)) return st;
        if (!get_map(&a.tmap_xs8, 2, a.xs, (uint64_t)a.rows_sf, NT_X, s13, 8, sps, &st)) return st;
        if (!get_map(&a.tmap_hs8, 2, a.hs, (uint64_t)a.rows_sf, NT_H, s2, 8, sps, &st)) return st;
    }
    // the first kernel of the forward clears the device error word (a memset here would break the
    // programmatic-dependent-launch chain between the permutation and the gather)
    return from_cuda(launch_forward(a, s));
}

moe_status_t moe_mxfp4_forward(const moe_layer_desc *d, const uint16_t *d_x, const void *d_packed,
                               const float *d_topk_w, const int32_t *d_offsets, const int32_t *d_padded_offsets,
                               const int32_t *d_row_to_pair, void *d_y, void *d_workspace, size_t workspace_bytes,
                               void *stream)
{
    return moe_mxfp4_forward_timed(d, d_x, d_packed, d_topk_w, d_offsets, d_padded_offsets, d_row_to_pair, d_y,
                                   d_workspace, workspace_bytes, nullptr, stream);
}

moe_status_t moe_read_device_error(void *d_error_word, int *code, void *stream)
{
    if (!d_error_word || !code) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    int v = 0;
    if (cudaMemcpyAsync(&v, d_error_word, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemsetAsync(d_error_word, 0, sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
    *code = v;
    return MOE_OK;
}

}  // extern "C"

// Expert parallelism: the two data-movement steps around the expert GEMMs when the
// experts of one layer are split over G ranks in contiguous ranges of E/G.
//
// The layer is the one of "DeepSeek V4 Flash 单卡 MI300X" (txtmix.com) §一 and §三
// (top-k routing, grouped MXFP4 expert GEMMs, routing-weighted combine); the
// pages run it on one GPU and do not shard it. Here each rank routes its own
// tokens, sends every (token, slot) pair's activation row to the rank owning the
// pair's expert, runs the grouped GEMMs on the rows it received for its own
// experts (k = 1, weight 1: the per-pair expert outputs), gets the outputs of its
// pairs back and combines them in slot order, which is the single-GPU combine.
//
// Send order: pairs sorted by (expert, token), i.e. the unpadded order of the
// stable permutation. Rank g's experts [g*EPR, (g+1)*EPR) then form one
// contiguous run of that order, offsets[g*EPR] .. offsets[(g+1)*EPR], so the
// all-to-all needs no further sorting; the outputs come back in the same order.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/moe_mxfp4.h"
#include "moe_internal.h"

namespace moe {
namespace {

// Expert e with offsets[e] <= i < offsets[e + 1] (the last such e when experts are empty).
__device__ __forceinline__ int expert_of(const int32_t *offsets, int E, int64_t i)
{
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(offsets + mid) <= i) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Send row i (of the P pairs in expert-major, token-ascending order): the bf16 activation row of the
// pair's token, 16 bytes per thread, and the pair's expert as an id local to its owner.
__global__ void ep_pack_kernel(const uint16_t *__restrict__ x, int H, int E, int k, int epr, int64_t P,
                               const int32_t *__restrict__ offsets, const int32_t *__restrict__ padded,
                               const int32_t *__restrict__ row_to_pair, uint16_t *__restrict__ send_x,
                               int32_t *__restrict__ send_ids)
{
    griddep_wait();
    const int cpr = H / 8;                                  // 16-byte chunks per row
    const int64_t n = P * cpr;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = idx / cpr;
        const int c = (int)(idx - i * cpr);
        const int e = expert_of(offsets, E, i);
        const int32_t p = __ldg(row_to_pair + __ldg(padded + e) + (i - __ldg(offsets + e)));
        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + (int64_t)(p / k) * H) + c);
        reinterpret_cast<uint4 *>(send_x + i * H)[c] = v;
        if (c == 0) send_ids[i] = e % epr;
    }
}

// y[t] = sum_j w[t, j] * returned[pos(t, j)], slots ascending, pos(p) = offsets[e] + pair_to_row[p] -
// padded[e] for the pair's expert e: where the pair's row went in the send order. A pair without a row
// (pair_to_row < 0) or with an expert outside [0, E) adds nothing and is recorded in *err.
__global__ void ep_combine_kernel(const float *__restrict__ ret, int T, int H, int E, int k,
                                  const int32_t *__restrict__ ids, const float *__restrict__ w,
                                  const int32_t *__restrict__ offsets, const int32_t *__restrict__ padded,
                                  const int32_t *__restrict__ pair_to_row, float *__restrict__ y, int32_t *err)
{
    griddep_wait();
    const int vec = H / 4;
    const int64_t n = (int64_t)T * vec;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < n; idx += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = idx / vec;
        const int c4 = (int)(idx - t * vec);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const int64_t p = t * k + j;
            const int e = __ldg(ids + p);
            const int32_t row = __ldg(pair_to_row + p);
            if (e < 0 || e >= E || row < 0) {
                if (c4 == 0 && err) atomicCAS(err, 0, DEV_ERR_ID_RANGE);
                continue;
            }
            const int64_t pos = (int64_t)__ldg(offsets + e) + (row - __ldg(padded + e));
            const float wj = __ldg(w + p);
            const float4 s = __ldg(reinterpret_cast<const float4 *>(ret + pos * H) + c4);
            acc.x = fmaf(wj, s.x, acc.x);
            acc.y = fmaf(wj, s.y, acc.y);
            acc.z = fmaf(wj, s.z, acc.z);
            acc.w = fmaf(wj, s.w, acc.w);
        }
        reinterpret_cast<float4 *>(y + t * H)[c4] = acc;
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int grid_for(int64_t n)
{
    int64_t g = (n + 255) / 256;
    if (g > 8 * 1024) g = 8 * 1024;
    return g < 1 ? 1 : (int)g;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_ep_dispatch_pack(const uint16_t *d_x, int T, int H, int E, int k, int experts_per_rank,
                                             const int32_t *d_offsets, const int32_t *d_padded_offsets,
                                             const int32_t *d_row_to_pair, uint16_t *d_send_x,
                                             int32_t *d_send_local_ids, void *stream)
{
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E || experts_per_rank <= 0) return MOE_ERR_INVALID_ARG;
    if (E % experts_per_rank || H % 8 || E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    const void *ptrs[] = {d_x, d_offsets, d_padded_offsets, d_row_to_pair, d_send_x, d_send_local_ids};
    for (const void *p : ptrs)
        if (!p) return MOE_ERR_INVALID_ARG;
    for (const void *p : ptrs)
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    const int64_t P = (int64_t)T * k;
    cudaError_t e = launch_ex(ep_pack_kernel, dim3(grid_for(P * (H / 8))), dim3(256), 0, (cudaStream_t)stream, true,
                              d_x, H, E, k, experts_per_rank, P, d_offsets, d_padded_offsets, d_row_to_pair, d_send_x,
                              d_send_local_ids);
    note_launch(1);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status_t moe_ep_combine(const float *d_returned, int T, int H, int E, int k, const int32_t *d_topk_ids,
                                       const float *d_topk_w, const int32_t *d_offsets,
                                       const int32_t *d_padded_offsets, const int32_t *d_pair_to_row, float *d_y,
                                       int32_t *d_error, void *stream)
{
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || k > E) return MOE_ERR_INVALID_ARG;
    if (H % 4 || E > 1024 || k > 32) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    const void *ptrs[] = {d_returned, d_topk_ids, d_topk_w, d_offsets, d_padded_offsets, d_pair_to_row, d_y};
    for (const void *p : ptrs)
        if (!p) return MOE_ERR_INVALID_ARG;
    for (const void *p : ptrs)
        if (!aligned16(p)) return MOE_ERR_MISALIGNED;
    cudaError_t e = launch_ex(ep_combine_kernel, dim3(grid_for((int64_t)T * (H / 4))), dim3(256), 0,
                              (cudaStream_t)stream, true, d_returned, T, H, E, k, d_topk_ids, d_topk_w, d_offsets,
                              d_padded_offsets, d_pair_to_row, d_y, d_error);
    note_launch(1);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

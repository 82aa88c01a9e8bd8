// Per-expert histogram, prefix offsets, block-padded offsets and the stable
// token permutation, in one thread block.
//
// Method: "DeepSeek V4 Flash 单卡 MI300X" (txtmix.com) §三 — the expert
// histogram is built over a padded, block-aligned layout, and lanes past the
// logical block (here: past the warp's own range of real pairs, and past
// T*k) must be masked, or they inject non-existent expert indices into the
// routing (the page's fix masks with offs_local < BLOCK_SIZE in addition to
// the global bound). Every lane below carries that two-sided mask.
//
// Pairs p = t*k + j are split into nw <= 32 contiguous warp ranges (about 64
// pairs per warp, so a decode batch touches one or two histogram rows per
// expert instead of 32). Phase 1: each
// warp histograms its range into its own shared-memory row with
// __match_any_sync (one leader per distinct expert per 32 lanes). Phase 2:
// per expert, a scan over the warp rows turns counts into warp bases; a block
// scan over experts gives offsets and padded offsets. Phase 3: each warp walks
// its range again in order; a pair's row is padded[e] + warp base + (pairs of
// e earlier in the range), so rows of one expert come out in ascending pair
// order (stable). Phase 4 writes -1 into padding and tail rows.
//
// The fused routing + permutation kernel (small batches) runs the per-token
// routing of route_token.cuh in the same thread block first, so a decode
// step spends one launch on both.
#include <cstdint>

#include "moe_internal.h"
#include "route_token.cuh"

namespace moe {

constexpr int PERM_THREADS = 1024;
constexpr int PERM_WARPS = PERM_THREADS / 32;

// Inclusive block-wide scan of one int per thread (1024 threads).
__device__ __forceinline__ int block_inclusive_scan(int v, int *warp_tot)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_tot[wid] = v;
    __syncthreads();
    if (wid == 0) {
        int t = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xFFFFFFFFu, t, o);
            if (lane >= o) t += n;
        }
        warp_tot[lane] = t;
    }
    __syncthreads();
    int r = v + (wid > 0 ? warp_tot[wid - 1] : 0);
    __syncthreads();
    return r;
}

__device__ __forceinline__ void permute_block(const int32_t *__restrict__ ids, int T, int E, int k, int block_m,
                                              int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                                              int32_t *__restrict__ padded, int32_t *__restrict__ row_to_pair,
                                              int64_t rows_cap, int32_t *__restrict__ pair_to_row,
                                              int32_t *__restrict__ dev_error)
{
    extern __shared__ int smem[];
    int *hist = smem;                                  // [PERM_WARPS][E]
    int *cnt = hist + PERM_WARPS * E;                  // [E]
    int *pad_start = cnt + E;                          // [E + 1]
    int *warp_tot = pad_start + E + 1;                 // [32]
    __shared__ int s_err;

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t P = (int64_t)T * k;
    const int nw = (int)(P / 64 + 1 < PERM_WARPS ? P / 64 + 1 : PERM_WARPS);   // warps holding pairs
    const int64_t lo = wid < nw ? P * wid / nw : P, hi = wid < nw ? P * (wid + 1) / nw : P;
    const unsigned lt_mask = (1u << lane) - 1u;

    if (tid == 0) s_err = 0;
    for (int i = tid; i < nw * E; i += PERM_THREADS) hist[i] = 0;
    __syncthreads();

    // Phase 1: per-warp histogram; lanes past this warp's range are masked.
    int *my = hist + wid * E;
    for (int64_t base = lo; base < hi; base += 32) {
        int64_t p = base + lane;
        bool valid = p < hi;                           // logical-block mask (never past T*k)
        int e = valid ? ids[p] : -1;
        if (valid && (e < 0 || e >= E)) { e = -1; s_err = 1; }
        unsigned m = __match_any_sync(0xFFFFFFFFu, e);
        if (e >= 0 && (m & lt_mask) == 0u) my[e] += __popc(m);
        __syncwarp();                                  // next iteration's leader may be another lane
    }
    __syncthreads();

    // Phase 2: warp bases per expert, then offsets / padded offsets.
    int c = 0, pc = 0;
    for (int e = tid; e < E; e += PERM_THREADS) {      // E <= 1024: at most one expert per thread
        int run = 0;
        for (int w = 0; w < nw; ++w) {
            int v = hist[w * E + e];
            hist[w * E + e] = run;
            run += v;
        }
        cnt[e] = run;
        c = run;
        pc = (run + block_m - 1) / block_m * block_m;
    }
    int inc_c = block_inclusive_scan(tid < E ? c : 0, warp_tot);
    int inc_p = block_inclusive_scan(tid < E ? pc : 0, warp_tot);
    if (tid < E) {
        counts[tid] = c;
        offsets[tid + 1] = inc_c;
        padded[tid + 1] = inc_p;
        pad_start[tid + 1] = inc_p;
    }
    if (tid == 0) {
        offsets[0] = 0;
        padded[0] = 0;
        pad_start[0] = 0;
    }
    __syncthreads();

    // Phase 3: stable scatter.
    for (int64_t base = lo; base < hi; base += 32) {
        int64_t p = base + lane;
        bool valid = p < hi;
        int e = valid ? ids[p] : -1;
        if (valid && (e < 0 || e >= E)) e = -1;
        unsigned m = __match_any_sync(0xFFFFFFFFu, e);
        int before = (e >= 0) ? my[e] : 0;
        __syncwarp();
        if (e >= 0) {
            int row = pad_start[e] + before + __popc(m & lt_mask);
            row_to_pair[row] = (int32_t)p;
            pair_to_row[p] = row;
            if ((m & lt_mask) == 0u) my[e] = before + __popc(m);
        } else if (valid) {
            pair_to_row[p] = -1;
        }
        __syncwarp();
    }

    // Phase 4: padding rows of each expert, then the tail up to rows_cap.
    for (int e = tid; e < E; e += PERM_THREADS)
        for (int r = pad_start[e] + cnt[e]; r < pad_start[e + 1]; ++r) row_to_pair[r] = -1;
    for (int64_t r = pad_start[E] + tid; r < rows_cap; r += PERM_THREADS) row_to_pair[r] = -1;

    __syncthreads();
    if (tid == 0 && s_err && dev_error) atomicExch(dev_error, DEV_ERR_ID_RANGE);
}

__global__ void __launch_bounds__(PERM_THREADS, 1)
permute_kernel(const int32_t *__restrict__ ids, int T, int E, int k, int block_m,
               int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int32_t *__restrict__ padded,
               int32_t *__restrict__ row_to_pair, int64_t rows_cap, int32_t *__restrict__ pair_to_row,
               int32_t *__restrict__ dev_error)
{
    griddep_wait();                   // ids come from the kernel before (launched with pdl)
    griddep_launch_dependents();
    permute_block(ids, T, E, k, block_m, counts, offsets, padded, row_to_pair, rows_cap, pair_to_row, dev_error);
}

// Routing of all T tokens (warp w takes tokens w, w + 32, ...), then the
// permutation of the ids just written, in one thread block.
template <int VPL>
__global__ void __launch_bounds__(PERM_THREADS, 1)
route_permute_kernel(const float *__restrict__ logits, int T, int E, int k, int block_m, int32_t *__restrict__ ids,
                     float *__restrict__ w, uint32_t *__restrict__ bitmatrix, int32_t *__restrict__ counts,
                     int32_t *__restrict__ offsets, int32_t *__restrict__ padded, int32_t *__restrict__ row_to_pair,
                     int64_t rows_cap, int32_t *__restrict__ pair_to_row, int32_t *__restrict__ dev_error)
{
    // the gather launched next (with pdl) only waits on this grid, so it may start now
    griddep_launch_dependents();
    __shared__ int32_t s_ids[ROUTE_PERMUTE_FUSED_MAX_T * 32];    // this block's ids (k <= 32), read back by the permutation
    for (int t = threadIdx.x >> 5; t < T; t += PERM_WARPS)
        route_token<VPL>(logits, t, E, k, ids, w, bitmatrix, s_ids);
    __syncthreads();          // the ids written above are visible to the whole block
    permute_block(s_ids, T, E, k, block_m, counts, offsets, padded, row_to_pair, rows_cap, pair_to_row, dev_error);
}

static size_t permute_smem(int E) { return sizeof(int) * ((size_t)PERM_WARPS * E + E + E + 1 + 32); }

// Raise a kernel's dynamic shared-memory limit to what E = 1024 needs, once per device (bit d of *mask);
// the attribute is a per-function maximum, so smaller launches are unaffected.
template <typename Kern>
static cudaError_t allow_permute_smem(Kern kern, unsigned long long *mask)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 64 && ((__atomic_load_n(mask, __ATOMIC_RELAXED) >> dev) & 1ull)) return cudaSuccess;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)permute_smem(1024));
    if (err == cudaSuccess && dev < 64) __atomic_fetch_or(mask, 1ull << dev, __ATOMIC_RELAXED);
    return err;
}

template <int VPL>
static cudaError_t launch_fused(const float *logits, int T, int E, int k, int block_m, int32_t *ids, float *w,
                                uint32_t *bitmatrix, int32_t *counts, int32_t *offsets, int32_t *padded,
                                int32_t *row_to_pair, int64_t rows_cap, int32_t *pair_to_row, int32_t *dev_error,
                                cudaStream_t s)
{
    static unsigned long long attr_set = 0;
    const size_t smem = permute_smem(E);
    cudaError_t err = allow_permute_smem(route_permute_kernel<VPL>, &attr_set);
    if (err != cudaSuccess) return err;
    route_permute_kernel<VPL><<<1, PERM_THREADS, smem, s>>>(logits, T, E, k, block_m, ids, w, bitmatrix, counts,
                                                            offsets, padded, row_to_pair, rows_cap, pair_to_row,
                                                            dev_error);
    return cudaGetLastError();
}

cudaError_t launch_route_permute(const float *logits, int T, int E, int k, int block_m, int32_t *ids, float *w,
                                 uint32_t *bitmatrix, int32_t *counts, int32_t *offsets, int32_t *padded,
                                 int32_t *row_to_pair, int64_t rows_cap, int32_t *pair_to_row, int32_t *dev_error,
                                 cudaStream_t s)
{
    if (T > ROUTE_PERMUTE_FUSED_MAX_T) {       // routing wants many blocks: two launches
        cudaError_t err = launch_route(logits, T, E, k, ids, w, bitmatrix, s);
        if (err != cudaSuccess) return err;
        return launch_permute(ids, T, E, k, block_m, counts, offsets, padded, row_to_pair, rows_cap, pair_to_row,
                              dev_error, s);
    }
    const int vpl = (E + 31) / 32;
    cudaError_t err;
    if (vpl <= 1) err = launch_fused<1>(logits, T, E, k, block_m, ids, w, bitmatrix, counts, offsets, padded, row_to_pair, rows_cap, pair_to_row, dev_error, s);
    else if (vpl <= 2) err = launch_fused<2>(logits, T, E, k, block_m, ids, w, bitmatrix, counts, offsets, padded, row_to_pair, rows_cap, pair_to_row, dev_error, s);
    else if (vpl <= 4) err = launch_fused<4>(logits, T, E, k, block_m, ids, w, bitmatrix, counts, offsets, padded, row_to_pair, rows_cap, pair_to_row, dev_error, s);
    else if (vpl <= 8) err = launch_fused<8>(logits, T, E, k, block_m, ids, w, bitmatrix, counts, offsets, padded, row_to_pair, rows_cap, pair_to_row, dev_error, s);
    else if (vpl <= 16) err = launch_fused<16>(logits, T, E, k, block_m, ids, w, bitmatrix, counts, offsets, padded, row_to_pair, rows_cap, pair_to_row, dev_error, s);
    else err = launch_fused<32>(logits, T, E, k, block_m, ids, w, bitmatrix, counts, offsets, padded, row_to_pair, rows_cap, pair_to_row, dev_error, s);
    note_launch(1);
    return err;
}

cudaError_t launch_permute(const int32_t *ids, int T, int E, int k, int block_m, int32_t *counts,
                           int32_t *offsets, int32_t *padded, int32_t *row_to_pair, int64_t rows_cap,
                           int32_t *pair_to_row, int32_t *dev_error, cudaStream_t s)
{
    static unsigned long long attr_set = 0;
    const size_t smem = permute_smem(E);
    cudaError_t err = allow_permute_smem(permute_kernel, &attr_set);
    if (err != cudaSuccess) return err;
    err = launch_ex(permute_kernel, dim3(1), dim3(PERM_THREADS), smem, s, true, ids, T, E, k, block_m, counts,
                    offsets, padded, row_to_pair, rows_cap, pair_to_row, dev_error);
    note_launch(1);
    return err;
}

}  // namespace moe

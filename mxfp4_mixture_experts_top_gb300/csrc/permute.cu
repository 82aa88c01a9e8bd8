// Per-expert histogram, prefix offsets, block-padded offsets and the stable
// token permutation: one thread block for small batches, many above 4096
// (token, slot) pairs.
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

// ---------------------------------------------------------------------------------------------
// Multi-block permutation for large batches. Block b owns experts [8b, 8b + 8). Every block builds
// the histogram of all experts itself (the ids are a few hundred KB, read from L2), so it knows
// every padded start without a workspace or any wait on another block; block 0 writes counts,
// offsets and padded offsets. Then each block walks all pairs in chunks of PM_CHUNK and scatters
// the pairs of its own experts: warp w of a chunk takes PM_SUB runs of 32 consecutive pairs and
// ranks each pair among the earlier pairs of its expert in the warp with one ballot per owned
// expert; a scan over the warps per expert adds the earlier warps of the chunk and the earlier
// chunks. Rows come out in ascending pair order inside each expert segment, bit-identical to the
// one-block kernel. The same two-sided lane mask applies: a lane counts only if it is inside its
// run and below T*k. (__match_any_sync, whose cost grows with the number of distinct experts in a
// warp, is avoided here: the histogram uses plain shared-memory adds, which conflict only where
// lanes share an expert.)
constexpr int PM_EPB = 8;                        // experts per block
constexpr int PM_SUB = 8;                        // runs of 32 pairs per warp and chunk
constexpr int PM_CHUNK = PERM_THREADS * PM_SUB;  // pairs per chunk
// Above this many pairs the permutation runs on many blocks.
constexpr int64_t PERMUTE_MULTI_MIN_PAIRS = 4096;

__global__ void __launch_bounds__(PERM_THREADS, 1)
permute_multi_kernel(const int32_t *__restrict__ ids, int T, int E, int k, int block_m,
                     int32_t *__restrict__ counts, int32_t *__restrict__ offsets, int32_t *__restrict__ padded,
                     int32_t *__restrict__ row_to_pair, int64_t rows_cap, int32_t *__restrict__ pair_to_row,
                     int32_t *__restrict__ dev_error)
{
    griddep_wait();                   // ids come from the kernel before (launched with pdl)
    griddep_launch_dependents();
    extern __shared__ int smem[];
    int *cnt = smem;                           // [E]
    int *pad_start = cnt + E;                  // [E + 1]
    int *warp_tot = pad_start + E + 1;         // [32]
    __shared__ int wcnt[PERM_WARPS][PM_EPB];   // pairs of each local expert in each warp's runs
    __shared__ int wbase[PERM_WARPS][PM_EPB];  // rows before each warp's first pair of the expert
    __shared__ int run[PM_EPB];                // rows of the expert filled by earlier chunks
    __shared__ int s_err;

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int64_t P = (int64_t)T * k;
    const int e0 = blockIdx.x * PM_EPB;
    const int ne = E - e0 < PM_EPB ? E - e0 : PM_EPB;
    const unsigned lt_mask = (1u << lane) - 1u;

    for (int i = tid; i < E; i += PERM_THREADS) cnt[i] = 0;
    if (tid < PM_EPB) run[tid] = 0;
    if (tid == 0) s_err = 0;
    __syncthreads();

    // Phase A: histogram of all experts. The ids of the next chunk are loaded before the current
    // chunk is counted, so the loads of one chunk overlap the adds of the one before.
    int nxt[PM_SUB];
#pragma unroll
    for (int sub = 0; sub < PM_SUB; ++sub) {
        const int64_t p = (int64_t)sub * PERM_THREADS + tid;
        nxt[sub] = p < P ? __ldg(ids + p) : -1;
    }
    for (int64_t base = 0; base < P; base += PM_CHUNK) {
        int ev[PM_SUB];
#pragma unroll
        for (int sub = 0; sub < PM_SUB; ++sub) {
            ev[sub] = nxt[sub];
            const int64_t p = base + PM_CHUNK + (int64_t)sub * PERM_THREADS + tid;
            nxt[sub] = p < P ? __ldg(ids + p) : -1;
        }
#pragma unroll
        for (int sub = 0; sub < PM_SUB; ++sub) {
            const int64_t p = base + (int64_t)sub * PERM_THREADS + tid;
            const int e = ev[sub];
            if (p < P) {
                if (e >= 0 && e < E) {
                    atomicAdd(&cnt[e], 1);
                } else {
                    s_err = 1;
                    if (blockIdx.x == 0) pair_to_row[p] = -1;
                }
            }
        }
    }
    __syncthreads();

    // Phase B: offsets and padded offsets (E <= 1024: one expert per thread).
    const int c = tid < E ? cnt[tid] : 0;
    const int pc = (c + block_m - 1) / block_m * block_m;
    const int inc_c = block_inclusive_scan(c, warp_tot);
    const int inc_p = block_inclusive_scan(pc, warp_tot);
    if (tid < E) {
        pad_start[tid + 1] = inc_p;
        if (blockIdx.x == 0) {
            counts[tid] = c;
            offsets[tid + 1] = inc_c;
            padded[tid + 1] = inc_p;
        }
    }
    if (tid == 0) {
        pad_start[0] = 0;
        if (blockIdx.x == 0) {
            offsets[0] = 0;
            padded[0] = 0;
        }
    }
    __syncthreads();

    // Phase C: stable scatter of this block's experts, chunk by chunk (the next chunk's ids are
    // loaded while the current chunk is ranked). Lane j < PM_EPB keeps the warp's running count of
    // local expert j in this chunk.
#pragma unroll
    for (int sub = 0; sub < PM_SUB; ++sub) {
        const int64_t p = ((int64_t)wid * PM_SUB + sub) * 32 + lane;
        nxt[sub] = p < P ? __ldg(ids + p) : -1;
    }
    for (int64_t base = 0; base < P; base += PM_CHUNK) {
        int el_s[PM_SUB], rank_s[PM_SUB];
#pragma unroll
        for (int sub = 0; sub < PM_SUB; ++sub) {
            el_s[sub] = nxt[sub];
            const int64_t p = base + PM_CHUNK + ((int64_t)wid * PM_SUB + sub) * 32 + lane;
            nxt[sub] = p < P ? __ldg(ids + p) : -1;
        }
        int mine = 0;                                   // lane j: pairs of local expert j so far
#pragma unroll
        for (int sub = 0; sub < PM_SUB; ++sub) {
            const int e = el_s[sub];                    // -1 past T*k (the load above masks it)
            const int el = (e >= e0 && e < e0 + ne) ? e - e0 : -1;
            unsigned same = 0u;
            int add = 0;
#pragma unroll
            for (int j = 0; j < PM_EPB; ++j) {
                const unsigned b = __ballot_sync(0xFFFFFFFFu, el == j);
                if (el == j) same = b;
                if (lane == j) add = __popc(b);
            }
            const int before = __shfl_sync(0xFFFFFFFFu, mine, el >= 0 ? el : 0);
            el_s[sub] = el;
            rank_s[sub] = before + __popc(same & lt_mask);
            mine += add;
        }
        if (lane < PM_EPB) wcnt[wid][lane] = mine;
        __syncthreads();
        if (wid < ne) {                       // warp j scans local expert j over the 32 warps
            const int v = wcnt[lane][wid];
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += n;
            }
            const int r = run[wid];
            wbase[lane][wid] = r + incl - v;
            const int tot = __shfl_sync(0xFFFFFFFFu, incl, 31);
            __syncwarp();
            if (lane == 0) run[wid] = r + tot;
        }
        __syncthreads();
#pragma unroll
        for (int sub = 0; sub < PM_SUB; ++sub) {
            if (el_s[sub] >= 0) {
                const int64_t p = base + ((int64_t)wid * PM_SUB + sub) * 32 + lane;
                const int row = pad_start[e0 + el_s[sub]] + wbase[wid][el_s[sub]] + rank_s[sub];
                row_to_pair[row] = (int32_t)p;
                pair_to_row[p] = row;
            }
        }
    }

    // Phase D: padding rows of this block's experts; the tail up to rows_cap split over all blocks.
    for (int j = 0; j < ne; ++j) {
        const int e = e0 + j;
        for (int r = pad_start[e] + cnt[e] + tid; r < pad_start[e + 1]; r += PERM_THREADS) row_to_pair[r] = -1;
    }
    for (int64_t r = pad_start[E] + (int64_t)blockIdx.x * PERM_THREADS + tid; r < rows_cap;
         r += (int64_t)gridDim.x * PERM_THREADS)
        row_to_pair[r] = -1;
    __syncthreads();
    if (blockIdx.x == 0 && tid == 0 && s_err && dev_error) atomicExch(dev_error, DEV_ERR_ID_RANGE);
}

static size_t permute_smem(int E) { return sizeof(int) * ((size_t)PERM_WARPS * E + E + E + 1 + 32); }
static size_t permute_multi_smem(int E) { return sizeof(int) * ((size_t)E + E + 1 + 32); }

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
    if ((int64_t)T * k > PERMUTE_MULTI_MIN_PAIRS) {
        const int blocks = (E + PM_EPB - 1) / PM_EPB;
        cudaError_t err = launch_ex(permute_multi_kernel, dim3(blocks), dim3(PERM_THREADS), permute_multi_smem(E), s,
                                    true, ids, T, E, k, block_m, counts, offsets, padded, row_to_pair, rows_cap,
                                    pair_to_row, dev_error);
        note_launch(1);
        return err;
    }
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

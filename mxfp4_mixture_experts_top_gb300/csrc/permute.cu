// Per-expert histogram, prefix offsets, block-padded offsets and the stable
// token permutation: one thread block for small batches, many above 2048
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
// Chunked permutation for large batches, in three launches. The pairs are cut into nc chunks of C
// consecutive pairs (the last chunk also takes the remainder), with C a multiple of PC_THREADS and
// C >= E. Until the last launch overwrites it, chunk b's own slice of pair_to_row, entries
// [b*C, b*C + E), holds the chunk's per-expert numbers, so no workspace is needed:
//   1. chunk histograms (one block per chunk): slice[e] = pairs of expert e in the chunk;
//   2. per expert (one warp each), an exclusive scan over the chunks: slice[e] = pairs of e in the
//      earlier chunks; counts[e] = the total;
//   3. per chunk (one block each): offsets and padded offsets from the counts (block 0 writes them),
//      then the chunk's pairs in order, 256 at a time: a pair's row is padded[e] + (pairs of e in
//      earlier chunks) + (in earlier rounds of this chunk) + (in earlier warps of this round) +
//      (in earlier lanes of its warp). Rows of one expert come out in ascending pair order, the
//      same rows as the one-block kernel. Padding rows of experts b, b + nc, ... and a 1/nc share
//      of the tail get -1.
// The two-sided lane mask applies in launches 1 and 3: a lane counts only inside its chunk, which
// never extends past T*k.
constexpr int PC_THREADS = 256;
constexpr int PC_WARPS = PC_THREADS / 32;
constexpr int PC_TARGET_CHUNKS = 256;            // chunks are at least P / 256 pairs
// Above this many pairs the permutation runs chunked on many blocks.
constexpr int64_t PERMUTE_MULTI_MIN_PAIRS = 2048;

struct ChunkPlan {
    int64_t C;     // pairs per chunk (the last chunk: P - (nc - 1) * C)
    int nc;        // chunks
};

static ChunkPlan chunk_plan(int64_t P, int E)
{
    int64_t c = (P + PC_TARGET_CHUNKS - 1) / PC_TARGET_CHUNKS;
    if (c < E) c = E;
    c = (c + PC_THREADS - 1) / PC_THREADS * PC_THREADS;
    ChunkPlan pl;
    pl.C = c;
    pl.nc = (int)(P / c);          // 1 .. 256: P > 2048 and C <= max(1024, P / 256 + 256) < P; C >= P / 256
    return pl;
}

__device__ __forceinline__ void chunk_range(int64_t P, int64_t C, int nc, int b, int64_t &lo, int64_t &hi)
{
    lo = (int64_t)b * C;
    hi = b == nc - 1 ? P : lo + C;
}

__global__ void __launch_bounds__(PC_THREADS)
permute_chunk_hist_kernel(const int32_t *__restrict__ ids, int64_t P, int E, int64_t C, int nc,
                          int32_t *__restrict__ pair_to_row)
{
    griddep_wait();                   // ids come from the kernel before (launched with pdl)
    griddep_launch_dependents();
    extern __shared__ int smem[];
    int *hist = smem;                 // [E]
    int64_t lo, hi;
    chunk_range(P, C, nc, blockIdx.x, lo, hi);
    for (int e = threadIdx.x; e < E; e += PC_THREADS) hist[e] = 0;
    __syncthreads();
    for (int64_t p = lo + threadIdx.x; p < hi; p += PC_THREADS) {    // lanes past the chunk are masked
        const int e = __ldg(ids + p);
        if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += PC_THREADS) pair_to_row[lo + e] = hist[e];
}

__global__ void __launch_bounds__(PC_THREADS)
permute_chunk_scan_kernel(int E, int64_t C, int nc, int32_t *__restrict__ counts, int32_t *__restrict__ pair_to_row)
{
    griddep_wait();                   // the chunk histograms come from the kernel before
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int e = blockIdx.x * PC_WARPS + (threadIdx.x >> 5);
    if (e >= E) return;                                   // uniform per warp
    constexpr int MAXC = (PC_TARGET_CHUNKS + 31) / 32;     // chunks per lane (nc <= 256)
    const int c0 = lane * nc / 32, c1 = (lane + 1) * nc / 32;
    int v[MAXC];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
        v[i] = c0 + i < c1 ? pair_to_row[(int64_t)(c0 + i) * C + e] : 0;
        sum += v[i];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    int run = incl - sum;
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
        if (c0 + i < c1) pair_to_row[(int64_t)(c0 + i) * C + e] = run;
        run += v[i];
    }
    if (lane == 31) counts[e] = incl;
}

// Inclusive scan of one int per thread over a PC_THREADS block.
__device__ __forceinline__ int chunk_block_scan(int v, int *warp_tot)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xFFFFFFFFu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_tot[wid] = v;
    __syncthreads();
    if (wid == 0) {
        int t = lane < PC_WARPS ? warp_tot[lane] : 0;
#pragma unroll
        for (int o = 1; o < PC_WARPS; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, t, o);
            if (lane >= o) t += n;
        }
        if (lane < PC_WARPS) warp_tot[lane] = t;
    }
    __syncthreads();
    const int r = v + (wid > 0 ? warp_tot[wid - 1] : 0);
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(PC_THREADS)
permute_chunk_scatter_kernel(const int32_t *__restrict__ ids, int64_t P, int E, int block_m, int64_t C, int nc,
                             const int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                             int32_t *__restrict__ padded, int32_t *__restrict__ row_to_pair, int64_t rows_cap,
                             int32_t *__restrict__ pair_to_row, int32_t *__restrict__ dev_error)
{
    griddep_wait();                   // counts and the per-chunk bases come from the kernel before
    griddep_launch_dependents();
    extern __shared__ int smem[];
    int *pad_start = smem;                       // [E + 1]
    int *cnt = pad_start + E + 1;                // [E]
    int *base = cnt + E;                         // [E]: next row of expert e for this chunk
    int *wc = base + E;                          // [PC_WARPS][E]: pairs of e in each warp's 32 lanes
    __shared__ int warp_tot[32];
    __shared__ int s_err;

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const unsigned lt_mask = (1u << lane) - 1u;
    int64_t lo, hi;
    chunk_range(P, C, nc, blockIdx.x, lo, hi);

    // offsets and padded offsets: thread i scans experts 4i .. 4i+3 (E <= 1024)
    int c4[4], s_c = 0, s_p = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int e = tid * 4 + q;
        c4[q] = e < E ? __ldg(counts + e) : 0;
        s_c += c4[q];
        s_p += (c4[q] + block_m - 1) / block_m * block_m;
    }
    if (tid == 0) s_err = 0;
    const int inc_c = chunk_block_scan(s_c, warp_tot);
    const int inc_p = chunk_block_scan(s_p, warp_tot);
    {
        int rc = inc_c - s_c, rp = inc_p - s_p;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = tid * 4 + q;
            if (e < E) {
                pad_start[e] = rp;
                cnt[e] = c4[q];
                base[e] = rp + pair_to_row[lo + e];            // this chunk's slice: rows of e in earlier chunks
                if (blockIdx.x == 0) {
                    offsets[e] = rc;
                    padded[e] = rp;
                }
            }
            rc += c4[q];
            rp += (c4[q] + block_m - 1) / block_m * block_m;
        }
        if (tid == PC_THREADS - 1) {
            pad_start[E] = rp;
            if (blockIdx.x == 0) {
                offsets[E] = rc;
                padded[E] = rp;
            }
        }
    }
    for (int i = tid; i < PC_WARPS * E; i += PC_THREADS) wc[i] = 0;
    __syncthreads();                  // the slice has been read: its entries may now be overwritten

    for (int64_t r0 = lo; r0 < hi; r0 += PC_THREADS) {
        const int64_t p = r0 + tid;
        const bool valid = p < hi;                          // logical-block mask (never past T*k)
        int e = valid ? __ldg(ids + p) : -1;
        if (valid && (e < 0 || e >= E)) { e = -1; s_err = 1; }
        const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
        const bool leader = (m & lt_mask) == 0u;
        if (e >= 0 && leader) wc[wid * E + e] = __popc(m);
        __syncthreads();
        if (e >= 0) {
            int row = base[e] + __popc(m & lt_mask);
            for (int w = 0; w < wid; ++w) row += wc[w * E + e];
            row_to_pair[row] = (int32_t)p;
            pair_to_row[p] = row;
        } else if (valid) {
            pair_to_row[p] = -1;
        }
        __syncthreads();
        if (e >= 0 && leader) {
            atomicAdd(&base[e], __popc(m));
            wc[wid * E + e] = 0;
        }
        __syncthreads();
    }

    // padding rows of experts b, b + nc, ...; the tail up to rows_cap split over the blocks
    for (int e = blockIdx.x; e < E; e += nc)
        for (int r = pad_start[e] + cnt[e] + tid; r < pad_start[e + 1]; r += PC_THREADS) row_to_pair[r] = -1;
    for (int64_t r = pad_start[E] + (int64_t)blockIdx.x * PC_THREADS + tid; r < rows_cap;
         r += (int64_t)nc * PC_THREADS)
        row_to_pair[r] = -1;
    __syncthreads();
    if (tid == 0 && s_err && dev_error) atomicExch(dev_error, DEV_ERR_ID_RANGE);
}

static size_t chunk_scatter_smem(int E) { return sizeof(int) * ((size_t)E + 1 + E + E + (size_t)PC_WARPS * E); }
// launched without raising the dynamic shared memory limit: up to 1,024 experts must fit the default 48 KB
static_assert(sizeof(int) * (1024 + 1 + 1024 + 1024 + PC_WARPS * 1024) <= 48 * 1024,
              "chunk scatter shared memory at 1,024 experts exceeds the default limit");

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
    const int64_t P = (int64_t)T * k;
    if (P > PERMUTE_MULTI_MIN_PAIRS) {
        const ChunkPlan pl = chunk_plan(P, E);
        cudaError_t err = launch_ex(permute_chunk_hist_kernel, dim3(pl.nc), dim3(PC_THREADS), sizeof(int) * (size_t)E,
                                    s, true, ids, P, E, pl.C, pl.nc, pair_to_row);
        if (err != cudaSuccess) return err;
        err = launch_ex(permute_chunk_scan_kernel, dim3((E + PC_WARPS - 1) / PC_WARPS), dim3(PC_THREADS), 0, s, true,
                        E, pl.C, pl.nc, counts, pair_to_row);
        if (err != cudaSuccess) return err;
        err = launch_ex(permute_chunk_scatter_kernel, dim3(pl.nc), dim3(PC_THREADS), chunk_scatter_smem(E), s, true,
                        (const int32_t *)ids, P, E, block_m, pl.C, pl.nc, (const int32_t *)counts, offsets, padded,
                        row_to_pair, rows_cap, pair_to_row, dev_error);
        note_launch(3);
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

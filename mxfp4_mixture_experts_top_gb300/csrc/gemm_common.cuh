// Declarations shared by the grouped-GEMM kernels: the launch parameters, the
// tile list decode, the error word and the SiLU of the W13 epilogue.
#pragma once
#include <cuda.h>

#include <cstdint>

#include "moe_internal.h"

namespace moe {

constexpr int TMEM_COLS = 512;

struct GemmParams {
    CUtensorMap tm_a;         // weight nibbles, box 128 x (128 * SPS) rows
    CUtensorMap tm_a1;        // weight nibbles, box 128 x 128 rows (a stage that straddles two tiles)
    CUtensorMap tm_b, tm_b1;  // activation terms [K/128][NT][rows][128] bytes, box 128 x NMAX x NT x (SPS | 1) slabs
    CUtensorMap tm_bs, tm_bs1; // their scale words [K/128][NT][rows_sf] (uint32), box NMAX x NT x (SPS | 1)
    const uint8_t *wsf;       // this matrix's prepacked scale region
    const int32_t *offsets;   // [E+1]
    const int32_t *padded;    // [E+1]
    const int32_t *row_to_pair;
    int E, K, MB;             // MB: 128-row weight tiles per expert
    int I, H, k;
    float swiglu_limit;
    int64_t P, rows_cap, rows_sf;
    uint8_t *hq;              // W13 out: h terms [I/128][NTO][rows_cap][128]
    uint8_t *hs;              // W13 out: h term scale words [I/128][NTO][rows_sf], byte = K-block % 4
    float *staging;           // W2 out [P, H]
    float *y;                 // fast combine (weight-major W2 only): adds w[pair] * o into y[pair / k]; nullptr: staging
    const float *topk_w;      // [T, k], with y
    int32_t *dev_error;
};

__device__ __forceinline__ void record_error(int32_t *dev_error, int code)
{
    if (dev_error) atomicCAS(dev_error, 0, code);
}

// Tile t -> (expert, token block, weight row tile); tile_start is the
// exclusive prefix over experts of ceil(count / NMAX) * MB.
struct Tile {
    int e, mb, row0, n;
};

template <int NMAX>
__device__ __forceinline__ Tile decode_tile(int t, const int *tile_start, int E, int MB, const int *cnt,
                                            const int *pad0)
{
    int lo = 0, hi = E - 1;                 // largest e with tile_start[e] <= t
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
    }
    Tile r;
    r.e = lo;
    int local = t - tile_start[lo];
    int nb = local / MB;
    r.mb = local - nb * MB;
    int rem = cnt[lo] - nb * NMAX;
    int n = rem < NMAX ? rem : NMAX;
    r.n = (n + 15) & ~15;
    r.row0 = pad0[lo] + nb * NMAX;
    return r;
}

// decode_tile with the expert's row count and first padded row read from the permutation offsets in
// global memory (for kernels that keep only the tile prefix in shared memory)
template <int NMAX>
__device__ __forceinline__ Tile decode_tile_g(int t, const int *tile_start, int E, int MB, const int32_t *offsets,
                                              const int32_t *padded)
{
    int lo = 0, hi = E - 1;                 // largest e with tile_start[e] <= t
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= t) lo = mid; else hi = mid - 1;
    }
    Tile r;
    r.e = lo;
    int local = t - tile_start[lo];
    int nb = local / MB;
    r.mb = local - nb * MB;
    int rem = (__ldg(offsets + lo + 1) - __ldg(offsets + lo)) - nb * NMAX;
    int n = rem < NMAX ? rem : NMAX;
    r.n = (n + 15) & ~15;
    r.row0 = __ldg(padded + lo) + nb * NMAX;
    return r;
}

// SiLU(g) = g / (1 + e^-g) with the fast exp and divide (about 1e-6 relative error, far below the 8
// bits h keeps in its two terms). For g < -88, e^-g is +inf and the quotient is -0.
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// The decode GEMMs (16-row tiles, 8-row with rows8, at most 2 rows per expert) as one persistent launch (gemm_decode.cu):
// W13 tiles, then W2 tiles, each W2 tile of an expert after that expert's W13 tiles (counters done13[E],
// zeroed by the caller before). decode_fused_supported: the shapes it takes.
bool decode_fused_supported(int H, int I, int E);
cudaError_t launch_gemm_decode(const GemmParams &g13, const GemmParams &g2, uint32_t *done13, bool fast, bool rows8,
                               int grid, cudaStream_t s, bool pdl);

// Token-major tiles for large batches (gemm_rows.cu): 128 token rows x 256 weight rows per tile.
// MODE 0: W13, MODE 1: W2. p.MB must be even.
// Token-major tiles: 128 token rows per tile (stacked = false) or 64 token rows with their two terms
// stacked as the MMA's A rows (stacked = true); 256 weight rows either way (H % 256 == 0).
cudaError_t launch_gemm_rows(const GemmParams &p, int mode, bool stacked, int grid, cudaStream_t s, bool pdl);

}  // namespace moe

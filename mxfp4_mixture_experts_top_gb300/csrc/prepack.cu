// One-time reorder of canonical MXFP4 weights into the prepacked format of
// mxfp4_tile.cuh, and the inverse decode to dense bf16 (for checks).
//
// The gate/up pairing inside each W13 tile is the "gate/up interleave" layout
// the fused-SiLU kernel needs ("DeepSeek V4 Flash 单卡 MI300X" (txtmix.com),
// §三: mxfp4.fused-silu adds a gate/up interleave layout): a tile's epilogue
// finds gate(f) and up(f) in lanes i and i+16 of the same warp.
#include <cuda_bf16.h>

#include <cstdint>

#include "moe_internal.h"
#include "mxfp4_tile.cuh"

namespace moe {

size_t packed_w13_bytes(int E, int H, int I)
{
    return (size_t)E * (size_t)(2 * I / TILE_ROWS) * (size_t)(H / KSLAB) * (SLAB_NIB_BYTES + SLAB_SF_BYTES);
}

size_t packed_w2_bytes(int E, int H, int I)
{
    return (size_t)E * (size_t)(H / TILE_ROWS) * (size_t)(I / KSLAB) * (SLAB_NIB_BYTES + SLAB_SF_BYTES);
}

// One thread per (tile-slab block, tile row r, 16-byte chunk c): 16 nibble
// bytes and, for c == 0, the row's 4 scale bytes of the slab.
__global__ void prepack_kernel(const uint8_t *__restrict__ q, const uint8_t *__restrict__ s, int E, int rows,
                               int K, int is_w13, int I, uint8_t *__restrict__ nib, uint8_t *__restrict__ sf)
{
    const int tiles = rows / TILE_ROWS, slabs = K / KSLAB;
    const int64_t total = (int64_t)E * tiles * slabs * TILE_ROWS * 4;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(idx & 3);
        const int r = (int)((idx >> 2) % TILE_ROWS);
        const int64_t blk = idx / (4 * TILE_ROWS);           // (e, tile, slab)
        const int slab = (int)(blk % slabs);
        const int tile = (int)((blk / slabs) % tiles);
        const int e = (int)(blk / ((int64_t)slabs * tiles));
        const int src = is_w13 ? w13_src_row(tile, r, I) : w2_src_row(tile, r);
        const int64_t row_off = (int64_t)e * rows + src;
        const uint4 in = *reinterpret_cast<const uint4 *>(q + row_off * (K / 2) + (int64_t)slab * (KSLAB / 2) + c * 16);
        *reinterpret_cast<uint4 *>(nib + (blk * TILE_ROWS + r) * (KSLAB / 2) + c * 16) = in;
        if (c == 0) {
            const uint8_t *ss = s + row_off * (K / 32) + (int64_t)slab * 4;
            const uint32_t v = (uint32_t)ss[0] | ((uint32_t)ss[1] << 8) | ((uint32_t)ss[2] << 16) | ((uint32_t)ss[3] << 24);
            *reinterpret_cast<uint32_t *>(sf + blk * SLAB_SF_BYTES + sf_offset(r, 0)) = v;
        }
    }
}

cudaError_t launch_prepack(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                           const uint8_t *w2_s, int E, int H, int I, uint8_t *packed, cudaStream_t st)
{
    const int threads = 256, blocks = 4096;
    uint8_t *w13 = packed, *w2 = packed + packed_w13_bytes(E, H, I);
    const size_t w13_nib = (size_t)E * 2 * I * (H / 2), w2_nib = (size_t)E * H * (I / 2);
    prepack_kernel<<<blocks, threads, 0, st>>>(w13_q, w13_s, E, 2 * I, H, 1, I, w13, w13 + w13_nib);
    prepack_kernel<<<blocks, threads, 0, st>>>(w2_q, w2_s, E, H, I, 0, I, w2, w2 + w2_nib);
    note_launch(2);
    return cudaGetLastError();
}

// Decode one expert's prepacked matrix to canonical-order bf16: one thread
// per (tile, slab, tile row, 32-element K-block).
__global__ void dequant_kernel(const uint8_t *__restrict__ nib, const uint8_t *__restrict__ sf, int rows, int K,
                               int is_w13, int I, __nv_bfloat16 *__restrict__ out)
{
    const int tiles = rows / TILE_ROWS, slabs = K / KSLAB;
    const int64_t total = (int64_t)tiles * slabs * TILE_ROWS * 4;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int kb = (int)(idx & 3);
        const int r = (int)((idx >> 2) % TILE_ROWS);
        const int64_t blk = idx / (4 * TILE_ROWS);
        const int slab = (int)(blk % slabs);
        const int tile = (int)(blk / slabs);
        const uint4 qv = *reinterpret_cast<const uint4 *>(nib + (blk * TILE_ROWS + r) * (KSLAB / 2) + kb * 16);
        const uint32_t sc = sf[blk * SLAB_SF_BYTES + sf_offset(r, kb)];
        const int row = is_w13 ? w13_src_row(tile, r, I) : w2_src_row(tile, r);
        __nv_bfloat16 *dst = out + (int64_t)row * K + (int64_t)slab * KSLAB + kb * 32;
        const uint32_t w[4] = {qv.x, qv.y, qv.z, qv.w};
#pragma unroll
        for (int i = 0; i < 32; ++i)
            dst[i] = __float2bfloat16_rn(e2m1_times_e8m0((w[i >> 3] >> (4 * (i & 7))) & 0xFu, sc));
    }
}

cudaError_t launch_dequant(const uint8_t *packed, int which, int expert, int E, int H, int I, uint16_t *out,
                           cudaStream_t st)
{
    const int threads = 256, blocks = 1024;
    __nv_bfloat16 *o = reinterpret_cast<__nv_bfloat16 *>(out);
    if (which == 0) {
        const size_t nib_e = (size_t)2 * I * (H / 2), sf_e = (size_t)2 * I * (H / 32);
        const uint8_t *nib = packed + (size_t)expert * nib_e;
        const uint8_t *sf = packed + (size_t)E * nib_e + (size_t)expert * sf_e;
        dequant_kernel<<<blocks, threads, 0, st>>>(nib, sf, 2 * I, H, 1, I, o);
    } else {
        const uint8_t *base = packed + packed_w13_bytes(E, H, I);
        const size_t nib_e = (size_t)H * (I / 2), sf_e = (size_t)H * (I / 32);
        const uint8_t *nib = base + (size_t)expert * nib_e;
        const uint8_t *sf = base + (size_t)E * nib_e + (size_t)expert * sf_e;
        dequant_kernel<<<blocks, threads, 0, st>>>(nib, sf, H, I, 0, I, o);
    }
    note_launch(1);
    return cudaGetLastError();
}

}  // namespace moe

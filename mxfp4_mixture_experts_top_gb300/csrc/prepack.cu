// One-time reorder of canonical MXFP4 weights into the prepacked tile format
// (see mxfp4_tile.cuh), and the inverse decode to dense bf16 through the same
// on-chip decoder the GEMMs use.
//
// The gate/up pairing inside each W13 tile is the "gate/up interleave" layout
// the fused-SiLU kernel needs ("DeepSeek V4 Flash 单卡 MI300X" (txtmix.com),
// §三: mxfp4.fused-silu adds a gate/up interleave layout): a tile's epilogue
// finds gate(f) and up(f) in lanes i and i+16 of the same warp.
#include <cstdint>

#include "moe_internal.h"
#include "mxfp4_tile.cuh"

namespace moe {

size_t packed_w13_bytes(int E, int H, int I)
{
    return (size_t)E * (size_t)(2 * I / TILE_ROWS) * (size_t)(H / KSLAB) * TILE_BYTES;
}

size_t packed_w2_bytes(int E, int H, int I)
{
    return (size_t)E * (size_t)(H / TILE_ROWS) * (size_t)(I / KSLAB) * TILE_BYTES;
}

// One thread per (block, chunk c, tile row r): 16 nibble bytes and, for
// c == 0, the tile row's 4 scale bytes.
__global__ void prepack_kernel(const uint8_t *__restrict__ q, const uint8_t *__restrict__ s, int E, int rows,
                               int K, int is_w13, int I, uint8_t *__restrict__ out)
{
    const int tiles = rows / TILE_ROWS, slabs = K / KSLAB;
    const int64_t total = (int64_t)E * tiles * slabs * 4 * TILE_ROWS;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(idx % TILE_ROWS);
        const int c = (int)((idx / TILE_ROWS) % 4);
        const int64_t blk = idx / (4 * TILE_ROWS);          // (e, tile, slab)
        const int slab = (int)(blk % slabs);
        const int tile = (int)((blk / slabs) % tiles);
        const int e = (int)(blk / ((int64_t)slabs * tiles));
        const int src = is_w13 ? w13_src_row(tile, r, I) : w2_src_row(tile, r);
        const int64_t row_off = ((int64_t)e * rows + src);
        const uint4 in = *reinterpret_cast<const uint4 *>(q + row_off * (K / 2) + (int64_t)slab * (KSLAB / 2) + c * 16);
        uint4 o;
        o.x = repack_word(in.x);
        o.y = repack_word(in.y);
        o.z = repack_word(in.z);
        o.w = repack_word(in.w);
        uint8_t *dst = out + blk * TILE_BYTES;
        *reinterpret_cast<uint4 *>(dst + (c * TILE_ROWS + r) * 16) = o;
        if (c == 0) {
            const uint8_t *ss = s + row_off * (K / 32) + (int64_t)slab * 4;
            uint32_t v = (uint32_t)ss[0] | ((uint32_t)ss[1] << 8) | ((uint32_t)ss[2] << 16) | ((uint32_t)ss[3] << 24);
            *reinterpret_cast<uint32_t *>(dst + TILE_NIB_BYTES + r * 4) = v;
        }
    }
}

cudaError_t launch_prepack(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                           const uint8_t *w2_s, int E, int H, int I, uint8_t *packed, cudaStream_t st)
{
    const int threads = 256, blocks = 4096;
    prepack_kernel<<<blocks, threads, 0, st>>>(w13_q, w13_s, E, 2 * I, H, 1, I, packed);
    prepack_kernel<<<blocks, threads, 0, st>>>(w2_q, w2_s, E, H, I, 0, I, packed + packed_w13_bytes(E, H, I));
    note_launch(2);
    return cudaGetLastError();
}

// Decode one expert's prepacked matrix to canonical-order bf16: one thread
// per (tile, slab, chunk, tile row), 32 elements each.
__global__ void dequant_kernel(const uint8_t *__restrict__ packed, int rows, int K, int is_w13, int I,
                               uint16_t *__restrict__ out)
{
    const int tiles = rows / TILE_ROWS, slabs = K / KSLAB;
    const int64_t total = (int64_t)tiles * slabs * 4 * TILE_ROWS;
    for (int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(idx % TILE_ROWS);
        const int c = (int)((idx / TILE_ROWS) % 4);
        const int64_t blk = idx / (4 * TILE_ROWS);
        const int slab = (int)(blk % slabs);
        const int tile = (int)(blk / slabs);
        const uint8_t *src = packed + blk * TILE_BYTES;
        const uint4 qv = *reinterpret_cast<const uint4 *>(src + (c * TILE_ROWS + r) * 16);
        const uint32_t sc = src[TILE_NIB_BYTES + r * 4 + c];
        const uint32_t m1 = scale_mult_lo(sc), m2 = scale_mult_hi(sc);
        const bool big = sc > 128u;
        uint32_t words[16];
        decode_word(qv.x, m1, m2, big, words + 0);
        decode_word(qv.y, m1, m2, big, words + 4);
        decode_word(qv.z, m1, m2, big, words + 8);
        decode_word(qv.w, m1, m2, big, words + 12);
        const int row = is_w13 ? w13_src_row(tile, r, I) : w2_src_row(tile, r);
        uint4 *dst = reinterpret_cast<uint4 *>(out + (int64_t)row * K + (int64_t)slab * KSLAB + c * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(words[4 * v], words[4 * v + 1], words[4 * v + 2], words[4 * v + 3]);
    }
}

cudaError_t launch_dequant(const uint8_t *packed, int which, int expert, int E, int H, int I, uint16_t *out,
                           cudaStream_t st)
{
    const int threads = 256, blocks = 1024;
    if (which == 0) {
        const uint8_t *base = packed + (size_t)expert * (packed_w13_bytes(E, H, I) / E);
        dequant_kernel<<<blocks, threads, 0, st>>>(base, 2 * I, H, 1, I, out);
    } else {
        const uint8_t *base = packed + packed_w13_bytes(E, H, I) + (size_t)expert * (packed_w2_bytes(E, H, I) / E);
        dequant_kernel<<<blocks, threads, 0, st>>>(base, H, I, 0, I, out);
    }
    note_launch(1);
    return cudaGetLastError();
}

}  // namespace moe

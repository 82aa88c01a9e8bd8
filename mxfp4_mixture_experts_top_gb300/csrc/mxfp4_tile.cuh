// Prepacked MXFP4 weight format: the layout the block-scaled tensor-core GEMMs
// stream straight from HBM.
//
// Format (OCP Microscaling v1.0): an E2M1 element is s|e1|e0|m with value
// (-1)^s * m/2 for e == 0 and (-1)^s * 2^(e-1) * (1 + m/2) otherwise; an E8M0
// scale byte s is 2^(s-127); one scale covers 32 consecutive K elements.
//
// A weight matrix [rows, K] is cut into A-tiles of 128 rows and K-slabs of
// KSLAB = 128 elements. Per matrix the packed buffer holds two regions:
//   nibbles  [tile][slab][128 tile rows][64 B]: each tile row's 128 elements of
//            the slab in canonical byte order (element 2i in the low nibble of
//            byte i). Viewed as a 2-D tensor of 128-element rows, consecutive
//            slabs of one tile are consecutive 128-row blocks, so one TMA box
//            of 128 * n rows fetches n slabs. The TMA "16 x U4, 16-byte
//            aligned" element type expands each 8-byte group to 16 bytes in
//            shared memory, which is the operand layout of tcgen05
//            kind::mxf8f6f4 for E2M1.
//   scales   [tile][slab][512 B]: byte (r % 32) * 16 + (r / 32) * 4 + kb holds
//            the scale of tile row r for the slab's K-block kb (0..3). Word c
//            of lane r0 (bytes r0 * 16 + 4c ..) is then exactly the tensor
//            memory cell (lane r0, column c) of the scale-factor operand: row
//            r0 + 32c, K-block kb in byte kb.
// The byte count equals the canonical MXFP4 bytes (nibbles + scales).
//
// W13 row tiles pair gate and up rows: tile row r = 32g + i holds feature
// f = 64*tile + 16g + (i % 16), the gate row (canonical row f) for i < 16
// and the up row (canonical row I + f) for i >= 16. W2 row tiles are plain:
// tile row r is canonical row 128*tile + r.
#pragma once
#include <cstdint>

namespace moe {

constexpr int KSLAB = 128;                                 // K elements per slab
constexpr int TILE_ROWS = 128;                             // A-tile rows (MMA M)
constexpr int SLAB_NIB_BYTES = TILE_ROWS * KSLAB / 2;      // 8192
constexpr int SLAB_SF_BYTES = TILE_ROWS * KSLAB / 32;      // 512
constexpr int SLAB_SMEM_BYTES = TILE_ROWS * 128;           // 16384: the slab expanded to 16 B per 16 elements

// Canonical source row of tile row r for W13 (features 64 per tile) or W2.
__host__ __device__ __forceinline__ int w13_src_row(int tile, int r, int I)
{
    int g = r >> 5, i = r & 31;
    int f = tile * 64 + g * 16 + (i & 15);
    return (i < 16) ? f : I + f;
}

__host__ __device__ __forceinline__ int w2_src_row(int tile, int r) { return tile * TILE_ROWS + r; }

// Offset of (tile row r, K-block kb) inside a slab's 512 scale bytes.
__host__ __device__ __forceinline__ int sf_offset(int r, int kb) { return (r & 31) * 16 + (r >> 5) * 4 + kb; }

// Exact E2M1 x E8M0 product as an fp32 (the power of two is built from its
// bits; products with |value| above the fp32 range become infinities, like
// any conversion of them to fp32 or bf16).
__device__ __forceinline__ float e2m1_times_e8m0(uint32_t code, uint32_t s)
{
    const uint32_t mag = code & 7u;
    const float m = mag == 0 ? 0.f : (mag == 1 ? 0.5f : (float)(2 + (mag & 1)) * (float)(1u << ((mag >> 1) - 1)) * 0.5f);
    const int e = (int)s - 127;
    const float p = e >= -126 ? __int_as_float((e + 127) << 23) : __int_as_float(1 << 22);   // 2^e, e >= -127
    const float v = m * p;
    return (code & 8u) ? -v : v;
}

}  // namespace moe

// Prepacked MXFP4 tile format and the on-chip E2M1 x E8M0 -> bf16 decoder.
//
// Format (OCP Microscaling v1.0): an E2M1 element is s|e1|e0|m with value
// (-1)^s * m/2 for e == 0 and (-1)^s * 2^(e-1) * (1 + m/2) otherwise; an E8M0
// scale byte s is 2^(s-127); one scale covers 32 consecutive K elements.
//
// Prepacked layout. A weight matrix is cut into A-tiles of 128 rows and
// K-slabs of KSLAB = 128 elements. Each (expert, row tile, slab) is one
// contiguous block of TILE_BYTES = 8704 bytes, fetched by one bulk copy:
//   [0, 8192)     nibbles: for chunk c in 0..3 (32 elements each), for tile
//                 row r in 0..127: 16 bytes. Warp lanes reading chunk c of
//                 rows 32g..32g+31 touch 512 consecutive bytes (no bank
//                 conflicts).
//   [8192, 8704)  scales: for tile row r: 4 bytes (chunks 0..3).
// Inside a 16-byte chunk, 32-bit word w (elements 8w..8w+7) stores element
// 8w+2j in nibble j and element 8w+2j+1 in nibble j+4 (j = 0..3), so one
// shift-and-mask yields a bf16x2 pair in natural K order.
//
// W13 row tiles pair gate and up rows: tile row r = 32g + i holds feature
// f = 64*tile + 16g + (i % 16), the gate row (canonical row f) for i < 16
// and the up row (canonical row I + f) for i >= 16. W2 row tiles are plain:
// tile row r is canonical row 128*tile + r.
#pragma once
#include <cstdint>

namespace moe {

constexpr int KSLAB = 128;                    // K elements per prepacked block
constexpr int TILE_ROWS = 128;                // A-tile rows (MMA M)
constexpr int TILE_NIB_BYTES = TILE_ROWS * KSLAB / 2;   // 8192
constexpr int TILE_SCALE_BYTES = TILE_ROWS * KSLAB / 32; // 512
constexpr int TILE_BYTES = TILE_NIB_BYTES + TILE_SCALE_BYTES;  // 8704

// Canonical source row of tile row r for W13 (features 64 per tile) or W2.
__host__ __device__ __forceinline__ int w13_src_row(int tile, int r, int I)
{
    int g = r >> 5, i = r & 31;
    int f = tile * 64 + g * 16 + (i & 15);
    return (i < 16) ? f : I + f;
}

__host__ __device__ __forceinline__ int w2_src_row(int tile, int r) { return tile * TILE_ROWS + r; }

// Repack one canonical 32-bit word (4 bytes, elements 2b in the low nibble and
// 2b+1 in the high nibble of byte b) into the decoder's nibble order.
__host__ __device__ __forceinline__ uint32_t repack_word(uint32_t src)
{
    uint32_t out = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        uint32_t byte = (src >> (8 * b)) & 0xFFu;
        out |= (byte & 0xFu) << (4 * b);          // element 8w+2b   -> nibble b
        out |= (byte >> 4) << (16 + 4 * b);       // element 8w+2b+1 -> nibble b+4
    }
    return out;
}

// bf16x2 multiplier that turns the raw pattern below into value * 2^(s-127).
// The raw pattern of magnitude code c is c << 6, i.e. the bf16 number
// e2m1(c) * 2^-126 (exponent field c >> 1, top mantissa bit c & 1; code 1 is
// the subnormal 2^-127 = 0.5 * 2^-126). Multiplying by 2^(s-1) is exact for
// s <= 128; larger scales take a second exact multiply (see decode_word).
__device__ __forceinline__ uint32_t scale_mult_lo(uint32_t s)
{
    uint32_t e = (s <= 128u) ? (s + 126u) : 253u;  // 2^(s-1) or 2^126
    uint32_t b = e << 7;
    return b | (b << 16);
}

__device__ __forceinline__ uint32_t scale_mult_hi(uint32_t s)
{
    uint32_t b = ((s <= 128u) ? 127u : s) << 7;    // 1.0 or 2^(s-127)
    return b | (b << 16);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Decode one prepacked 32-bit word into 4 bf16x2 words (elements 8w..8w+7 in
// order). `m1` = scale_mult_lo(s); `m2` = scale_mult_hi(s) is applied only
// when `big_scale` (s > 128 somewhere in the warp).
// Word j takes nibbles j and j+4. For j = 0, 1 they sit at bits 4j and 16+4j
// of q; for j = 2, 3 the same positions of q >> 8. Masking one pair and
// multiplying by 2^(6-4j') + 2^(12-4j') (j' = j mod 2) places each magnitude
// at bits 8..6 / 24..22 and each sign at bit 15 / 31 without carries; the
// final mask drops the other copies.
__device__ __forceinline__ void decode_word(uint32_t q, uint32_t m1, uint32_t m2, bool big_scale,
                                            uint32_t *out)
{
    const uint32_t q2 = q >> 8;
    uint32_t raw[4];
    raw[0] = ((q & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;
    raw[1] = ((q & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;
    raw[2] = ((q2 & 0x000F000Fu) * 0x1040u) & 0x81C081C0u;
    raw[3] = ((q2 & 0x00F000F0u) * 0x0104u) & 0x81C081C0u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        uint32_t r = bf16x2_mul(raw[j], m1);
        if (big_scale) r = bf16x2_mul(r, m2);
        out[j] = r;
    }
}

}  // namespace moe

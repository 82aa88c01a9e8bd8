// Grouped MXFP4 expert GEMMs for large batches: token-major tiles on tcgen05
// block-scaled MMAs (sm_103a).
//
// Method: "DeepSeek V4 Flash 单卡 MI300X" (txtmix.com) §三 — grouped MXFP4
// expert GEMMs with SiLU(gate)*up fused into the W13 epilogue, then W2; §九 —
// the optional SwiGLU clamp. Same arithmetic as gemm.cu; another tile shape.
//
// When experts hold hundreds of token rows the weight-major tiles of gemm.cu
// (128 weight rows x up to 96 token rows, all activation terms stacked along
// N) re-read every token row's terms once per 128 weight rows, and the SMs'
// operand intake from L2 bounds the tensor pipe. Here a tile is
//   A = 128 token rows of ONE activation term (E4M3, M = 128),
//   B = 256 weight rows (two prepacked 128-row tiles of E2M1, N = 256),
// and the terms are summed by the tensor core itself: for every 32-K block the
// MMA issuer runs one MMA per term into the same accumulator, both reading the
// same weight slab. Per useful multiply-add the SM then takes in
// 2 terms x 1 B / 256 + 0.5 B / 128 bytes, against 0.5 / 96 + 2 / 128 for the
// weight-major tile: about 1.8 times less.
//   * Stages are one 128-K slab: the activation box (128 rows x 2 terms,
//     32 KB) and the two weight slabs (expanded to 32 KB) with their scales.
//   * The accumulator is 128 lanes x 256 fp32 columns; with the scale-factor
//     cells it leaves no room for a second buffer, so the MMA issuer waits for
//     the epilogue to have read the previous tile (eight epilogue warps, each
//     reading its half of the columns in two 64-column chunks and releasing the
//     accumulator after its second load) while the producers keep filling the
//     rings with the next tile's slabs.
//   * W13 epilogue: a TMEM lane is one token row; columns 32g .. 32g+31 hold
//     the gate (first 16) and up (last 16) of features 128*nb + 16g + 0..15 (the
//     prepacked gate/up interleave), so SiLU(gate)*up and the 32-feature
//     block maximum of h are thread-local. h leaves as two MXFP8 terms in the
//     row-major term layout W2 reads.
//   * W2 epilogue: the thread's token row gets 256 consecutive output features
//     of its (token, slot) pair in the fp32 staging rows.
//   * Tile list (built on the device from the permutation offsets): expert,
//     then 128-row token block, then 256-row weight block. Rows of a block past
//     the expert's own rows (the next expert's, or the unwritten tail) are
//     computed and never stored.
// Stacked tiles (17 to 64 rows per expert, where 128 token rows would leave
// most of a tile empty; block-scaled MMAs take M = 128 only): a tile is 64
// token rows, and the A operand's 128 rows are their two terms, term 0 in rows
// 0-63 and term 1 in rows 64-127 (the order in which the 64-row activation box
// lands), so one MMA per 32-K block covers both terms and an activation slab
// still serves 256 weight rows. Lane quarters 0-1 of the accumulator then hold
// term 0's partial sums and quarters 2-3 term 1's, for the same tokens and
// columns; warps q and q ^ 2 trade 16-column pieces through shared memory and
// each finishes one 64-column chunk. Four weight and four activation stages.
// Warp roles (512 threads): 0-3 and 12-15 epilogue (columns 0-127 and
// 128-255 of lane quarter warp % 4), 4-7 scale-factor copiers, 8 MMA issuer
// and TMEM owner, 9 activation producer, 10 weight producer, 11 idle.
// Every wait is bounded (2 s); on time-out a CTA records MOE_ERR_TIMEOUT,
// drains its copies and MMAs, frees TMEM and exits.
#include <cuda_bf16.h>

#include <cstdint>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "mxfp4_tile.cuh"
#include "mxfp8_terms.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

// MODE 0: W13, MODE 1: W2. NW / NX: weight / activation ring stages; NSF: TMEM scale-factor cells.
// STACK: 64 token rows per tile, their two terms stacked as the MMA's 128 A rows (see above).
template <int MODE_, int NW_, int NX_, int NSF_, int EMAX_, bool STACK_ = false>
struct RCfg {
    static constexpr int MODE = MODE_, NW = NW_, NX = NX_, NSF = NSF_, EMAX = EMAX_;
    static constexpr bool STACK = STACK_;
    static constexpr int TM = STACK ? 64 : 128;      // token rows per tile
    static constexpr int MM = 128;                   // MMA M (A rows)
    static constexpr int TN = 256;                   // weight rows per tile
    static constexpr int NT = 2;                     // activation terms (x: NT_X; h: the Huge h terms)
    static constexpr int CELL_COLS = 16;             // one slab: A cells of term 0 and 1 (4 each), B (8)
    static constexpr int SF_BASE = TN;               // after the accumulator
    static constexpr int THREADS = 512;
    static constexpr int ND = 8;                     // done ring (see gemm.cu)
    static_assert(NW <= ND && NX <= ND && NSF <= ND, "done ring");
    static_assert(SF_BASE + NSF * CELL_COLS <= TMEM_COLS, "TMEM budget");
};

constexpr int NTH_HUGE = 2;
static_assert(NTH_HUGE == 2 && NT_X == 2, "the token-major tiles take two terms of x and of h");

using W13Rows = RCfg<0, 3, 3, 4, 1024>;
using W2Rows = RCfg<1, 3, 3, 4, 1024>;
using W13Rows64 = RCfg<0, 4, 4, 4, 1024, true>;
using W2Rows64 = RCfg<1, 4, 4, 4, 1024, true>;

template <class C>
struct RSmem {
    static constexpr int XTERM = C::TM * 128;                  // one term's rows of one slab
    static constexpr int XSTAGE = C::NT * XTERM;               // 32 KB (16 KB stacked: the A operand)
    static constexpr int WSTAGE = 2 * SLAB_SMEM_BYTES;         // two expanded weight slabs, 32 KB
    static constexpr int XSSTAGE = C::NT * C::TM * 4;          // scale words [term][row], 1 KB
    static constexpr int WSSTAGE = 2 * SLAB_SF_BYTES;          // 1 KB
    static constexpr int X_OFF = 0;
    static constexpr int W_OFF = X_OFF + C::NX * XSTAGE;
    static constexpr int XS_OFF = W_OFF + C::NW * WSTAGE;
    static constexpr int WS_OFF = XS_OFF + C::NX * XSSTAGE;
    // stacked tiles: per epilogue warp 16 columns x 32 lanes of fp32 partial sums for its partner
    static constexpr int EX_OFF = WS_OFF + C::NW * WSSTAGE;
    static constexpr int EX_BYTES = C::STACK ? 8 * 16 * 32 * 4 : 0;
    static constexpr int BAR_OFF = EX_OFF + EX_BYTES;
    static constexpr int NBARS = C::NW + C::NX + C::NSF + C::ND + 3;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int PREFIX_OFF = MISC_OFF + 16;
    // the tile prefix [E + 1] and the scan scratch [32] (an expert's rows are read from global memory)
    static constexpr size_t bytes(int E) { return 1024 + PREFIX_OFF + sizeof(int) * (size_t)(E + 1 + 32); }
    static_assert(XSTAGE % 1024 == 0 && WSTAGE % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static_assert(bytes(C::EMAX) <= 232448, "shared memory per CTA");
};

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1) moe_gemm_rows_kernel(const __grid_constant__ GemmParams p)
{
    constexpr int MODE = C::MODE, TM = C::TM, NT = C::NT;
    using S = RSmem<C>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *xring = smem + S::X_OFF;
    uint8_t *wring = smem + S::W_OFF;
    uint8_t *xsring = smem + S::XS_OFF;
    uint8_t *wsring = smem + S::WS_OFF;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::BAR_OFF);
    uint64_t *w_full = bars, *x_full = w_full + C::NW, *sf_full = x_full + C::NX;
    uint64_t *done = sf_full + C::NSF;
    uint64_t *d_full = done + C::ND, *d_empty = d_full + 1, *mma_done = d_empty + 1;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + S::MISC_OFF);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + S::MISC_OFF + 4);
    int *tile_start = reinterpret_cast<int *>(smem + S::PREFIX_OFF);
    int *scan_tmp = tile_start + p.E + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E, NBT = p.MB / 2;     // 256-row weight blocks per expert

    // ---- tile prefix over experts (E <= 1024: two experts per thread)
    {
        int v[2];
        int s = 0;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int e = tid * 2 + q;
            const int cnt = e < E ? (__ldg(p.offsets + e + 1) - __ldg(p.offsets + e)) : 0;
            v[q] = (cnt + TM - 1) / TM * NBT;
            s += v[q];
        }
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) scan_tmp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = lane < C::THREADS / 32 ? scan_tmp[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (lane >= o) w += n;
            }
            if (lane < C::THREADS / 32) scan_tmp[lane] = w;
        }
        __syncthreads();
        int run = incl - s + (warp > 0 ? scan_tmp[warp - 1] : 0);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int e = tid * 2 + q;
            if (e < E) tile_start[e] = run;
            run += v[q];
        }
        if (tid == C::THREADS - 1) tile_start[E] = run;
        __syncthreads();
    }
    const int total = tile_start[E];
    if ((int)blockIdx.x >= total) {           // uniform: this CTA has no tiles
        griddep_wait();
        return;
    }

    // ---- barriers and TMEM
    if (tid == 0) {
        for (int i = 0; i < C::NW; ++i) ptx::mbar_init(&w_full[i], 1);
        for (int i = 0; i < C::NX; ++i) ptx::mbar_init(&x_full[i], 1);
        for (int i = 0; i < C::NSF; ++i) ptx::mbar_init(&sf_full[i], 4);
        for (int i = 0; i < C::ND; ++i) ptx::mbar_init(&done[i], 1);
        ptx::mbar_init(d_full, 1);
        ptx::mbar_init(d_empty, 8);           // one arrival per epilogue warp
        ptx::mbar_init(mma_done, 1);
        *s_abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 8) {
        ptx::tmem_alloc(s_tmem, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int slabs = p.K / KSLAB;
    const int my_tiles = (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1;
    const int n_stages = my_tiles * slabs;      // one slab per stage
    const uint64_t LIM = WAIT_LIMIT_NS;

    auto fail = [&]() {
        *s_abort = 1;
        record_error(p.dev_error, DEV_ERR_TIMEOUT);
    };
    auto wait_done = [&](int q) -> bool {
        return q < 0 || ptx::mbar_wait(&done[q % C::ND], (uint32_t)((q / C::ND) & 1), s_abort, LIM);
    };
    auto tile_of = [&](int j) {
        return decode_tile_g<TM>((int)blockIdx.x + j * (int)gridDim.x, tile_start, E, NBT, p.offsets, p.padded);
    };

    if (warp == 10) {
        // ===================== weight producer: per slab the two 128-row weight tiles' E2M1 slabs (one
        // TMA box each, expanded in shared memory) and their scales (one bulk copy each)
        if (ptx::elect_one()) ptx::prefetch_tmap(&p.tm_a1);
        __syncwarp();
        int wi = 0;
        long long issued = 0;
        bool ok = true;
        int j = 0, ka = 0;
        Tile tl = tile_of(0);
        for (int s = 0; s < n_stages; ++s) {
            if (!__all_sync(0xFFFFFFFFu, wait_done(s - C::NW))) { ok = false; break; }
            if (ptx::elect_one()) {
                ptx::mbar_arrive_expect_tx(&w_full[wi], (uint32_t)(2 * (SLAB_NIB_BYTES + SLAB_SF_BYTES)));
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int mt = tl.e * p.MB + 2 * tl.mb + u;       // prepacked 128-row tile
                    const int r0 = (mt * slabs + ka) * TILE_ROWS;
                    ptx::tma_load_2d(wring + wi * S::WSTAGE + u * SLAB_SMEM_BYTES, &p.tm_a1, 0, r0, &w_full[wi]);
                    ptx::bulk_g2s(wsring + wi * S::WSSTAGE + u * SLAB_SF_BYTES,
                                  p.wsf + (size_t)(r0 / TILE_ROWS) * SLAB_SF_BYTES, SLAB_SF_BYTES, &w_full[wi]);
                }
            }
            __syncwarp();
            ++issued;
            if (++ka == slabs) {
                ka = 0;
                if (++j < my_tiles) tl = tile_of(j);
            }
            if (++wi == C::NW) wi = 0;
        }
        if (!ok && lane == 0) fail();
        volatile int never = 0;
        for (long long i = 1; i <= (issued < C::NW ? issued : C::NW); ++i) {
            const long long n = issued - i;
            __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&w_full[n % C::NW], (uint32_t)((n / C::NW) & 1), &never, LIM));
        }
    } else if (warp == 9) {
        // ===================== activation producer: per slab one 4-D box of both terms' 128 token rows and
        // one 3-D box of their scale words. The terms come from the kernel before (gather, or W13 for
        // W2): this warp waits for it; everything above and the weight stream may run earlier.
        if (ptx::elect_one()) {
            ptx::prefetch_tmap(&p.tm_b1);
            ptx::prefetch_tmap(&p.tm_bs1);
        }
        griddep_wait();
        if (lane == 0) griddep_launch_dependents();
        __syncwarp();
        int xi = 0;
        long long issued = 0;
        bool ok = true;
        int j = 0, ka = 0;
        Tile tl = tile_of(0);
        for (int s = 0; s < n_stages; ++s) {
            if (!__all_sync(0xFFFFFFFFu, wait_done(s - C::NX))) { ok = false; break; }
            if (ptx::elect_one()) {
                ptx::mbar_arrive_expect_tx(&x_full[xi], (uint32_t)(S::XSTAGE + S::XSSTAGE));
                ptx::tma_load_4d(xring + xi * S::XSTAGE, &p.tm_b1, 0, tl.row0, 0, ka, &x_full[xi]);
                ptx::tma_load_3d(xsring + xi * S::XSSTAGE, &p.tm_bs1, tl.row0, 0, ka, &x_full[xi]);
            }
            __syncwarp();
            ++issued;
            if (++ka == slabs) {
                ka = 0;
                if (++j < my_tiles) tl = tile_of(j);
            }
            if (++xi == C::NX) xi = 0;
        }
        if (!ok && lane == 0) fail();
        volatile int never = 0;
        for (long long i = 1; i <= (issued < C::NX ? issued : C::NX); ++i) {
            const long long n = issued - i;
            __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&x_full[n % C::NX], (uint32_t)((n / C::NX) & 1), &never, LIM));
        }
    } else if (warp >= 4 && warp < 8) {
        // ===================== scale-factor copiers: per slab one 16-column cell in this warp's lane
        // quarter: columns 0-3 term 0's token rows, 4-7 term 1's (row r at lane r % 32, column r / 32),
        // 8-15 the 256 weight rows (the prepacked 512-byte scale blocks are already in that order)
        int wi = 0, xi = 0, sc = 0;
        uint32_t wph = 0, xph = 0;
        bool ok = true;
        const uint32_t quarter = (uint32_t)((warp & 3) * 32) << 16;
        for (int s = 0; s < n_stages; ++s) {
            if (!__all_sync(0xFFFFFFFFu, wait_done(s - C::NSF) && ptx::mbar_wait(&w_full[wi], wph, s_abort, LIM) &&
                                             ptx::mbar_wait(&x_full[xi], xph, s_abort, LIM))) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t *xs = reinterpret_cast<const uint32_t *>(xsring + xi * S::XSSTAGE);
            const uint4 w0 = *reinterpret_cast<const uint4 *>(wsring + wi * S::WSSTAGE + lane * 16);
            const uint4 w1 = *reinterpret_cast<const uint4 *>(wsring + wi * S::WSSTAGE + SLAB_SF_BYTES + lane * 16);
            uint32_t vb[8];
            vb[0] = w0.x; vb[1] = w0.y; vb[2] = w0.z; vb[3] = w0.w;
            vb[4] = w1.x; vb[5] = w1.y; vb[6] = w1.z; vb[7] = w1.w;
            const uint32_t cell = tmem + quarter + (uint32_t)(C::SF_BASE + sc * C::CELL_COLS);
            if constexpr (C::STACK) {
                // A row 32c + lane is word 32c + lane of the stage ([term][64 rows]): columns 0-1 term 0,
                // 2-3 term 1
                ptx::tmem_st_32x32b_x4(cell, xs[lane], xs[32 + lane], xs[64 + lane], xs[96 + lane]);
            } else {
                uint32_t va[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) va[c] = xs[(c >> 2) * TM + lane + 32 * (c & 3)];
                ptx::tmem_st_32x32b_x8(cell, va);
            }
            ptx::tmem_st_32x32b_x8(cell + 8u, vb);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sf_full[sc]);
            if (++wi == C::NW) { wi = 0; wph ^= 1u; }
            if (++xi == C::NX) { xi = 0; xph ^= 1u; }
            if (++sc == C::NSF) sc = 0;
        }
        if (!ok && lane == 0) fail();
    } else if (warp == 8) {
        // ===================== MMA issuer: per slab, for each 32-K block, one MMA per term into the
        // tile's accumulator (A: the term's 128 token rows, B: the 256 weight rows, both K-major with
        // the 128-byte swizzle), then one commit freeing the slab's stages; at a tile's end a commit to
        // d_full. Before a tile's first MMA the epilogue must have read the previous tile.
        const uint64_t xdesc0 = ptx::smem_desc_sw128(ptx::smem_u32(xring));
        const uint64_t wdesc0 = ptx::smem_desc_sw128(ptx::smem_u32(wring));
        int wi = 0, xi = 0, sc = 0, ka = 0;
        uint32_t sph = 0, dph = 0;
        bool ok = true;
        for (int s = 0; s < n_stages && ok; ++s) {
            if (ka == 0) {
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(d_empty, dph ^ 1u, s_abort, LIM))) { ok = false; break; }
                ptx::tc_fence_after();
            }
            if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&sf_full[sc], sph, s_abort, LIM))) { ok = false; break; }
            ptx::tc_fence_after();
            if (ptx::elect_one()) {
                const uint32_t cell = tmem + (uint32_t)(C::SF_BASE + sc * C::CELL_COLS);
                const uint64_t wd = wdesc0 + (uint64_t)((uint32_t)(wi * S::WSTAGE) >> 4);
#pragma unroll
                for (int kb = 0; kb < 4; ++kb) {
                    if constexpr (C::STACK) {
                        // both terms in one MMA: A rows 0-63 term 0, 64-127 term 1 of the same tokens
                        const uint64_t xd = xdesc0 + (uint64_t)((uint32_t)(xi * S::XSTAGE) >> 4);
                        ptx::mma_mx_ss(tmem, xd + (uint64_t)(kb * 2), wd + (uint64_t)(kb * 2),
                                       ptx::idesc_mx(0u, 5u, C::MM, C::TN, (uint32_t)kb), cell, cell + 8u,
                                       (ka > 0 || kb > 0) ? 1u : 0u);
                    } else {
#pragma unroll
                        for (int t = 0; t < NT; ++t) {
                            const uint64_t xd = xdesc0 + (uint64_t)((uint32_t)(xi * S::XSTAGE + t * S::XTERM) >> 4);
                            ptx::mma_mx_ss(tmem, xd + (uint64_t)(kb * 2), wd + (uint64_t)(kb * 2),
                                           ptx::idesc_mx(0u, 5u, C::MM, C::TN, (uint32_t)kb), cell + (uint32_t)(4 * t),
                                           cell + 8u, (ka > 0 || kb > 0 || t > 0) ? 1u : 0u);
                        }
                    }
                }
                ptx::mma_commit(&done[s % C::ND]);
                if (ka == slabs - 1) ptx::mma_commit(d_full);
            }
            __syncwarp();
            if (++ka == slabs) {
                ka = 0;
                dph ^= 1u;
            }
            if (++wi == C::NW) wi = 0;
            if (++xi == C::NX) xi = 0;
            if (++sc == C::NSF) { sc = 0; sph ^= 1u; }
        }
        if (!ok && lane == 0) fail();
        volatile int never = 0;
        if (ptx::elect_one()) ptx::mma_commit(mma_done);
        __syncwarp();
        __all_sync(0xFFFFFFFFu, ptx::mbar_wait(mma_done, 0, &never, LIM));
    } else if (warp < 4 || warp >= 12) {
        // ===================== epilogue: lane quarter q = warp % 4, columns 128g .. 128g+127 (g = 0 for
        // warps 0-3, 1 for warps 12-15) in two chunks of 64. Token-row tiles: lane quarter q is token rows
        // 32q .. 32q+31 and the warp finishes both chunks. Stacked tiles: quarters 0-1 hold term 0 of token
        // rows 0-63 and quarters 2-3 term 1 of the same rows, so warps q and q ^ 2 hold the two halves of
        // the same sums: each sends the partner its partial sums of one chunk through shared memory, in four
        // rounds of 16 columns, and finishes the other (chunk q >> 1), term 0 + term 1 in both.
        const int q = warp & 3, g = warp >= 12 ? 1 : 0;
        const uint32_t t_lane = (uint32_t)(q * 32) << 16;
        const int trow = C::STACK ? (q & 1) * 32 + lane : q * 32 + lane;   // token row in the tile
        float *ex_send = reinterpret_cast<float *>(smem + S::EX_OFF) + (g * 4 + q) * 16 * 32;
        const float *ex_recv = reinterpret_cast<const float *>(smem + S::EX_OFF) + (g * 4 + (q ^ 2)) * 16 * 32;
        const uint32_t pair_bar = 1u + (uint32_t)(2 * g + (q & 1));        // named barrier of warps q, q ^ 2
        uint32_t dph = 0;
        bool ok = true;

        // W13: columns c0 .. c0+63 are features 128*nb + c0/2 + 0..31 (column groups c0/32 and c0/32 + 1),
        // one W2 K-block: SiLU(gate)*up, its block maximum and its NT terms; the terms' scale bytes are
        // returned in sb
        auto w13_chunk = [&](const Tile &tl, int64_t row, int c0, const uint32_t (&a0)[32], const uint32_t (&a1)[32],
                             uint32_t (&sb)[NT]) {
            const float L = p.swiglu_limit;
            float h[32];
            float mx = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float gt = __uint_as_float(a0[i]), up = __uint_as_float(a0[16 + i]);
                float gt2 = __uint_as_float(a1[i]), up2 = __uint_as_float(a1[16 + i]);
                if (L > 0.f) {
                    gt = fminf(gt, L);
                    up = fminf(fmaxf(up, -L), L);
                    gt2 = fminf(gt2, L);
                    up2 = fminf(fmaxf(up2, -L), L);
                }
                h[i] = silu_f(gt) * up;
                h[16 + i] = silu_f(gt2) * up2;
                mx = fmaxf(mx, fmaxf(fabsf(h[i]), fabsf(h[16 + i])));
            }
            const int e1 = mxfp8_block_exp(mx);
            const int blk = c0 >> 6;                   // K-block of the slab (0..3)
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                uint32_t w[8];
                sb[t] = 0;
#pragma unroll
                for (int z = 0; z < 8; ++z) {
                    const uint32_t lo = mxfp8_term_pair(h[4 * z], h[4 * z + 1], e1, t, sb[t]);
                    const uint32_t hi = mxfp8_term_pair(h[4 * z + 2], h[4 * z + 3], e1, t, sb[t]);
                    w[z] = lo | (hi << 16);
                }
                ptx::st_global_v8(p.hq + (((int64_t)tl.mb * NT + t) * p.rows_cap + row) * 128 + blk * 32, w);
            }
        };
        // W2: 256 contiguous bytes of the pair's staging row, in 32-byte stores (the combine reads them
        // back once, after the whole launch)
        auto w2_chunk = [&](const Tile &tl, int pair, int c0, const uint32_t (&a0)[32], const uint32_t (&a1)[32]) {
            float *dst = p.staging + (int64_t)pair * p.H + (int64_t)tl.mb * C::TN + c0;
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                uint32_t v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = a0[8 * z + u];
                ptx::st_global_v8_stream(dst + 8 * z, v);
            }
#pragma unroll
            for (int z = 0; z < 4; ++z) {
                uint32_t v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = a1[8 * z + u];
                ptx::st_global_v8_stream(dst + 32 + 8 * z, v);
            }
        };

        for (int j = 0; j < my_tiles; ++j) {
            const Tile tl = tile_of(j);
            ok = ok && __all_sync(0xFFFFFFFFu, ptx::mbar_wait(d_full, dph, s_abort, LIM));
            ptx::tc_fence_after();
            const bool row_ok = trow < tl.n;
            const int64_t row = (int64_t)tl.row0 + trow;
            int pair = -1;
            if (MODE == 1 && row_ok) {
                pair = __ldg(p.row_to_pair + row);
                if (pair >= p.P) {
                    record_error(p.dev_error, DEV_ERR_ID_RANGE);
                    pair = -1;
                }
            }
            if constexpr (C::STACK) {
                const int ch = q >> 1, c0 = 128 * g + 64 * ch, cs = 128 * g + 64 * (ch ^ 1);
                uint32_t a0[32], a1[32];
                // round r: the partner's columns cs + 16r go into this warp's slot (column-major,
                // lane-consecutive words), this warp's own columns c0 + 16r come from TMEM, and the
                // partner's term is added from its slot
                auto exchange_round = [&](int r, uint32_t (&own)[16]) {
                    __syncwarp();                            // the loads below are warp-collective
                    if (ok) {
                        uint32_t snd[16];
                        ptx::tmem_ld_32x32b_x16(tmem + t_lane + (uint32_t)(cs + 16 * r), snd);
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) ex_send[i * 32 + lane] = __uint_as_float(snd[i]);
                        ptx::tmem_ld_32x32b_x16(tmem + t_lane + (uint32_t)(c0 + 16 * r), own);
                        ptx::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) own[i] = 0u;
                    }
                    if (r == 3) {                            // the accumulator has been read
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (ok && lane == 0) ptx::mbar_arrive(d_empty);
                    }
                    ptx::bar_sync_n(pair_bar, 64);          // the partner's partial sums are in its slot
                    if (ok) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            own[i] = __float_as_uint(__uint_as_float(own[i]) + ex_recv[i * 32 + lane]);
                    }
                    ptx::bar_sync_n(pair_bar, 64);          // both slots read: they may be refilled
                };
                exchange_round(0, *reinterpret_cast<uint32_t (*)[16]>(a0));
                exchange_round(1, *reinterpret_cast<uint32_t (*)[16]>(a0 + 16));
                exchange_round(2, *reinterpret_cast<uint32_t (*)[16]>(a1));
                exchange_round(3, *reinterpret_cast<uint32_t (*)[16]>(a1 + 16));
                if (ok && row_ok) {
                    if (MODE == 0) {
                        uint32_t sb[NT];
                        w13_chunk(tl, row, c0, a0, a1, sb);
#pragma unroll
                        for (int t = 0; t < NT; ++t)         // byte 2g + ch of the row's scale word per term
                            p.hs[(((int64_t)tl.mb * NT + t) * p.rows_sf + row) * 4 + 2 * g + ch] = (uint8_t)sb[t];
                    } else if (pair >= 0) {
                        w2_chunk(tl, pair, c0, a0, a1);
                    }
                }
            } else {
                uint32_t sbytes[NT] = {0u, 0u};             // W13: this warp's two scale bytes per term
                for (int ch = 0; ch < 2; ++ch) {
                    const int c0 = 128 * g + 64 * ch;        // first column of the chunk
                    uint32_t a0[32], a1[32];
                    __syncwarp();                            // the loads below are warp-collective
                    if (ok) {
                        ptx::tmem_ld_32x32b_x32(tmem + t_lane + (uint32_t)c0, a0);
                        ptx::tmem_ld_32x32b_x32(tmem + t_lane + (uint32_t)(c0 + 32), a1);
                        ptx::tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) a0[i] = a1[i] = 0u;
                    }
                    if (ch == 1) {                            // the accumulator has been read
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (ok && lane == 0) ptx::mbar_arrive(d_empty);
                    }
                    if (!ok || !row_ok) continue;           // (re-converges at the __syncwarp above)
                    if (MODE == 0) {
                        uint32_t sb[NT];
                        w13_chunk(tl, row, c0, a0, a1, sb);
#pragma unroll
                        for (int t = 0; t < NT; ++t) sbytes[t] |= sb[t] << (8 * ch);
                    } else if (pair >= 0) {
                        w2_chunk(tl, pair, c0, a0, a1);
                    }
                }
                if (MODE == 0 && ok && row_ok) {
                    // K-blocks 2g and 2g + 1 of slab nb: bytes 2g, 2g + 1 of the row's scale word per term
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        uint16_t *ds = reinterpret_cast<uint16_t *>(p.hs + (((int64_t)tl.mb * NT + t) * p.rows_sf + row) * 4) + g;
                        *ds = (uint16_t)sbytes[t];
                    }
                }
            }
            dph ^= 1u;
        }
        if (!ok && lane == 0) fail();
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 8) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

template <class C>
cudaError_t launch_rows(const GemmParams &p, int grid, cudaStream_t s, bool pdl)
{
    static unsigned long long attr_set = 0;   // bit d: attribute set on device d
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !((attr_set >> dev) & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(moe_gemm_rows_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)RSmem<C>::bytes(C::EMAX));
        if (e != cudaSuccess) return e;
        if (dev < 64) __atomic_fetch_or(&attr_set, 1ull << dev, __ATOMIC_RELAXED);
    }
    return launch_ex(moe_gemm_rows_kernel<C>, dim3(grid), dim3(C::THREADS), RSmem<C>::bytes(p.E), s, pdl, p);
}

}  // namespace

cudaError_t launch_gemm_rows(const GemmParams &p, int mode, bool stacked, int grid, cudaStream_t s, bool pdl)
{
    if (stacked) return mode == 0 ? launch_rows<W13Rows64>(p, grid, s, pdl) : launch_rows<W2Rows64>(p, grid, s, pdl);
    return mode == 0 ? launch_rows<W13Rows>(p, grid, s, pdl) : launch_rows<W2Rows>(p, grid, s, pdl);
}

}  // namespace moe

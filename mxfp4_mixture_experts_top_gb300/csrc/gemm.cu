// Grouped MXFP4 expert GEMMs on tcgen05 (sm_103a), plus the gather and the
// routing-weighted combine.
//
// Method: "DeepSeek V4 Flash 单卡 MI300X" (txtmix.com) §三 — grouped MXFP4
// expert GEMMs, W13 with SiLU(gate)*up fused into its epilogue over a gate/up
// interleaved weight layout, then W2; §九 — the optional SwiGLU clamp. The
// combine y[t] = sum_j w[t,j] o_j is the routing-weighted scatter back to
// token order.
//
// Design (swap-AB, weights as the tcgen05 A operand in TMEM):
//   * A = 128 weight rows x K. MXFP4 tiles stream HBM -> shared memory by
//     1-D bulk copies (8704 B per 128 x 128 slab); 8 converter warps decode
//     E2M1 x E8M0 to exact bf16 in registers and write them straight into
//     tensor memory with tcgen05.st, so the dequantised operand never touches
//     shared memory (shared-memory bandwidth stays free for B).
//   * B = the expert's N token rows (N <= 192 for W13, <= 128 for W2, a
//     multiple of 16) loaded by 2-D TMA with the 128-byte swizzle.
//   * D = fp32 accumulator in TMEM, double-buffered so the epilogue of one
//     tile overlaps the main loop of the next.
//   * One elected thread issues tcgen05.mma kind::f16 (M=128, N, K=16);
//     completion is signalled with tcgen05.commit on mbarriers.
//   * Persistent CTAs (one per SM) walk a tile list built on the device from
//     the permutation offsets (no host synchronisation): expert-major, then
//     token block, then weight row tile, so concurrent CTAs share B tiles in
//     L2.
//   * W2 consumes the SiLU product as hi + lo bf16 terms (two MMAs into the
//     same accumulator), keeping ~16 bits of its precision.
// Warp roles (512 threads, every role warp-converged): 0-3 epilogue, 4 weight producer (bulk copies),
// 5 MMA issuer and TMEM owner, 6 activation producer (TMA), 7 idle, 8-15
// converters. Every wait is bounded (2 s); on
// time-out a CTA records MOE_ERR_TIMEOUT, drains its copies and MMAs, frees
// TMEM and exits.
#include <cuda_bf16.h>

#include <cstdint>

#include "moe_internal.h"
#include "mxfp4_tile.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int TMEM_COLS = 512;
constexpr int B_BOX_ROWS = 16;         // TMA box: 64 K elements (128 B) x 16 rows
constexpr int A_COLS = KSLAB / 2;      // TMEM columns per A buffer (bf16 pairs)

// Kernel configuration. MODE 0: W13 (activation rows -> SiLU(gate)*up),
// MODE 1: W2 ((h_hi, h_lo) rows -> per-pair outputs). NMAX: most token rows
// per tile (experts with more rows get several tiles). NB: activation ring
// slots (the token rows of one 128-K slab each), NW: weight ring slots (one
// 128 x 128 slab each), NA: TMEM A buffers, NACC: accumulators per tile (consecutive MMAs
// of a tile rotate over them and the epilogue sums them: with small N an MMA
// is short, and its latency rather than its work would otherwise set the
// pace). TMEM columns: 2 * NACC * NMAX for the
// double-buffered accumulators, then NA * 64 for the A buffers (<= 512).
template <int MODE_, int NMAX_, int NB_, int NW_, int NA_, int NACC_, int CONVW_>
struct Cfg {
    static constexpr int MODE = MODE_, NMAX = NMAX_, NB = NB_, NW = NW_, NA = NA_, NACC = NACC_;
    // converter warps (8 or 16) in groups of 8; group j takes the slabs i with
    // i % GROUPS == j, so the latency chains of GROUPS slabs overlap. In a
    // group, warp (g, part) decodes chunks 2*part, 2*part+1 of rows 32g..32g+31.
    static constexpr int GROUPS = CONVW_ / 8;
    static constexpr int THREADS = (8 + CONVW_) * 32;
    static_assert(CONVW_ == 8 || CONVW_ == 16, "converter warps");
    static constexpr int NOPS = MODE == 0 ? 1 : 2;
    static constexpr int D_COLS = NACC * NMAX;            // one accumulator set
    static constexpr int A_BASE = 2 * D_COLS;
    static_assert(A_BASE + NA * A_COLS <= TMEM_COLS, "TMEM budget");
    static_assert(NMAX % 16 == 0 && NMAX <= 256, "MMA N");
};

// Decode-sized tiles are bound by decoding MXFP4 at the HBM rate: 16
// converter warps, 6 A buffers. Prefill tiles are bound by the tensor pipe.
// decode, <= 2 rows per expert on average: 16-row tiles
using W13Tiny = Cfg<0, 16, 24, 12, 6, 2, 16>;
using W2Tiny = Cfg<1, 16, 12, 12, 6, 2, 16>;
// decode batches: <= 32 rows per tile
using W13Small = Cfg<0, 32, 12, 12, 6, 2, 16>;
using W2Small = Cfg<1, 32, 6, 12, 6, 2, 16>;
// mid: <= 64 rows per tile
using W13Mid = Cfg<0, 64, 6, 12, 4, 2, 16>;
using W2Mid = Cfg<1, 64, 3, 12, 4, 2, 16>;
// prefill: large tiles
using W13Large = Cfg<0, 192, 2, 8, 2, 1, 8>;
using W2Large = Cfg<1, 128, 2, 8, 4, 1, 8>;

struct GemmParams {
    CUtensorMap tm_b0;        // W13: gathered x; W2: h_hi
    CUtensorMap tm_b1;        // W2: h_lo
    const uint8_t *wpack;     // this matrix's prepacked tiles
    const int32_t *offsets;   // [E+1]
    const int32_t *padded;    // [E+1]
    const int32_t *row_to_pair;
    int E, K, MB;             // MB: 128-row weight tiles per expert
    int I, H, k;
    float swiglu_limit;
    int64_t P;
    __nv_bfloat16 *h_hi, *h_lo;   // W13 out [rows, I]
    float *staging;               // W2 out [P, H]
    int32_t *dev_error;
};

template <class C>
struct Smem {
    static constexpr int REGION = C::NMAX * 128;                 // one 64-K box column of NMAX rows
    static constexpr int BSTAGE = 2 * C::NOPS * REGION;            // [K half][operand][rows][128 B]
    static constexpr int B_OFF = 0;
    static constexpr int W_OFF = B_OFF + C::NB * BSTAGE;
    static constexpr int BAR_OFF = W_OFF + C::NW * TILE_BYTES;
    static constexpr int NBARS = 2 * C::NW + 2 * C::NB + 2 * C::NA + 2 * 2 + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int PREFIX_OFF = MISC_OFF + 16;
    static size_t bytes(int E) { return 1024 + PREFIX_OFF + sizeof(int) * (size_t)(E + 1 + 32); }
    static_assert(BSTAGE % 1024 == 0, "B stages must keep the 1024-byte swizzle alignment");
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

template <class C>
__device__ __forceinline__ Tile decode_tile(int t, const int *tile_start, int E, int MB,
                                            const int32_t *offsets, const int32_t *padded)
{
    constexpr int NMAX = C::NMAX;
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
    int count = __ldg(offsets + lo + 1) - __ldg(offsets + lo);
    int rem = count - nb * NMAX;
    int n = rem < NMAX ? rem : NMAX;
    r.n = (n + 15) & ~15;
    r.row0 = __ldg(padded + lo) + nb * NMAX;
    return r;
}

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1) moe_gemm_kernel(const __grid_constant__ GemmParams p)
{
    constexpr int MODE = C::MODE;
    using S = Smem<C>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *bring = smem + S::B_OFF;
    uint8_t *wring = smem + S::W_OFF;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::BAR_OFF);
    uint64_t *w_full = bars, *w_empty = w_full + C::NW;
    uint64_t *b_full = w_empty + C::NW, *b_empty = b_full + C::NB;
    uint64_t *a_full = b_empty + C::NB, *a_empty = a_full + C::NA;
    uint64_t *d_full = a_empty + C::NA, *d_empty = d_full + 2;
    uint64_t *mma_done = d_empty + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + S::MISC_OFF);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + S::MISC_OFF + 4);
    int *tile_start = reinterpret_cast<int *>(smem + S::PREFIX_OFF);
    int *scan_tmp = tile_start + p.E + 1;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E, MB = p.MB;

    // ---- tile prefix over experts (E <= 1024: two experts per thread)
    {
        int v[2];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            int e = tid * 2 + q;
            int cnt = e < E ? (__ldg(p.offsets + e + 1) - __ldg(p.offsets + e)) : 0;
            v[q] = (cnt + C::NMAX - 1) / C::NMAX * MB;
        }
        int s = v[0] + v[1];
        int incl = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += n;
        }
        if (lane == 31) scan_tmp[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = lane < C::THREADS / 32 ? scan_tmp[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int n = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (lane >= o) w += n;
            }
            if (lane < C::THREADS / 32) scan_tmp[lane] = w;
        }
        __syncthreads();
        int excl = incl - s + (warp > 0 ? scan_tmp[warp - 1] : 0);
        int e0 = tid * 2;
        if (e0 < E) tile_start[e0] = excl;
        if (e0 + 1 < E) tile_start[e0 + 1] = excl + v[0];
        if (e0 + 1 == E) tile_start[E] = excl + v[0];
        if (e0 + 2 == E) tile_start[E] = excl + v[0] + v[1];
        __syncthreads();
    }
    const int total = tile_start[E];
    if ((int)blockIdx.x >= total) return;     // uniform: this CTA has no tiles

    // ---- barriers and TMEM
    if (tid == 0) {
        for (int i = 0; i < C::NW; ++i) { ptx::mbar_init(&w_full[i], 1); ptx::mbar_init(&w_empty[i], 8); }
        for (int i = 0; i < C::NB; ++i) { ptx::mbar_init(&b_full[i], 1); ptx::mbar_init(&b_empty[i], 1); }
        for (int i = 0; i < C::NA; ++i) {
            ptx::mbar_init(&a_full[i], 8);
            ptx::mbar_init(&a_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&d_full[i], 1);
            ptx::mbar_init(&d_empty[i], 4);
        }
        ptx::mbar_init(mma_done, 1);
        *s_abort = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 5) {
        ptx::tmem_alloc(s_tmem, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const int slabs = p.K / KSLAB;
    constexpr int MMAS_PER_SLAB = 8 * C::NOPS;             // K = 128 in steps of 16, per operand
    const int nacc = slabs * MMAS_PER_SLAB < C::NACC ? slabs * MMAS_PER_SLAB : C::NACC;   // accumulators written
    const uint64_t LIM = WAIT_LIMIT_NS;

    auto fail = [&]() {
        *s_abort = 1;
        record_error(p.dev_error, DEV_ERR_TIMEOUT);
    };

    // Warps 4, 5 and 6 run their loops with all 32 lanes converged; one lane
    // issues each copy / MMA / commit (see ptx::elect_one).
    if (warp == 4) {
        // ===================== weight producer: one 8704-byte bulk copy per 128 x 128 slab
        int wi = 0;
        uint32_t wph = 0;
        long long issued = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            Tile tl = decode_tile<C>(t, tile_start, E, MB, p.offsets, p.padded);
            const uint8_t *wsrc = p.wpack + ((size_t)tl.e * MB + tl.mb) * (size_t)slabs * TILE_BYTES;
            for (int ka = 0; ka < slabs; ++ka) {
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&w_empty[wi], wph ^ 1u, s_abort, LIM))) { ok = false; break; }
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(&w_full[wi], TILE_BYTES);
                    ptx::bulk_g2s(wring + wi * TILE_BYTES, wsrc + (size_t)ka * TILE_BYTES, TILE_BYTES, &w_full[wi]);
                }
                __syncwarp();
                ++issued;
                if (++wi == C::NW) { wi = 0; wph ^= 1u; }
            }
        }
        if (!ok && lane == 0) fail();
        volatile int never = 0;
        // drain: every issued copy must land before shared memory is released
        for (long long i = 1; i <= (issued < C::NW ? issued : C::NW); ++i) {
            long long n = issued - i;
            __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&w_full[n % C::NW], (uint32_t)((n / C::NW) & 1), &never, LIM));
        }
    } else if (warp == 6) {
        // ===================== activation producer: the tile's token rows of one 128-K slab per
        // stage, as 2-D TMA boxes of 64 K x 16 rows
        if (ptx::elect_one()) {
            ptx::prefetch_tmap(&p.tm_b0);
            if (C::NOPS > 1) ptx::prefetch_tmap(&p.tm_b1);
        }
        __syncwarp();
        int bi = 0;
        uint32_t bph = 0;
        long long issued = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            Tile tl = decode_tile<C>(t, tile_start, E, MB, p.offsets, p.padded);
            const uint32_t bbytes = (uint32_t)(2 * C::NOPS * tl.n * 128);
            for (int ka = 0; ka < slabs; ++ka) {
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&b_empty[bi], bph ^ 1u, s_abort, LIM))) { ok = false; break; }
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(&b_full[bi], bbytes);
                    uint8_t *stage = bring + bi * S::BSTAGE;
                    for (int half = 0; half < 2; ++half) {
                        const int kx = ka * KSLAB + half * 64;
                        uint8_t *dst = stage + half * C::NOPS * S::REGION;
                        for (int r = 0; r < tl.n; r += B_BOX_ROWS)
                            ptx::tma_load_2d(dst + r * 128, &p.tm_b0, kx, tl.row0 + r, &b_full[bi]);
                        if (C::NOPS > 1)
                            for (int r = 0; r < tl.n; r += B_BOX_ROWS)
                                ptx::tma_load_2d(dst + S::REGION + r * 128, &p.tm_b1, kx, tl.row0 + r, &b_full[bi]);
                    }
                }
                __syncwarp();
                ++issued;
                if (++bi == C::NB) { bi = 0; bph ^= 1u; }
            }
        }
        if (!ok && lane == 0) fail();
        volatile int never = 0;
        for (long long i = 1; i <= (issued < C::NB ? issued : C::NB); ++i) {
            long long n = issued - i;
            __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&b_full[n % C::NB], (uint32_t)((n / C::NB) & 1), &never, LIM));
        }
    } else if (warp == 5) {
        // ===================== MMA issuer: per slab one A buffer, one activation stage
        const uint64_t bdesc_base = ptx::smem_desc_sw128(ptx::smem_u32(bring));   // stage 0, offset 0
        int ai = 0, bi = 0, di = 0;
        uint32_t aph = 0, bph = 0, dph = 0;
        bool ok = true, issued = false;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            Tile tl = decode_tile<C>(t, tile_start, E, MB, p.offsets, p.padded);
            const uint32_t idesc = ptx::idesc_bf16_f32(128, (uint32_t)tl.n);
            if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&d_empty[di], dph ^ 1u, s_abort, LIM))) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t dt0 = tmem + (uint32_t)(di * C::D_COLS);
            for (int ka = 0; ka < slabs; ++ka) {
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&a_full[ai], aph, s_abort, LIM) &&
                                                 ptx::mbar_wait(&b_full[bi], bph, s_abort, LIM))) { ok = false; break; }
                ptx::tc_fence_after();
                if (ptx::elect_one()) {
                    // All per-MMA offsets are compile-time constants off three per-slab bases;
                    // this warp shares its scheduler with busy converter warps, so every
                    // instruction here costs several cycles.
                    const uint32_t at0 = tmem + (uint32_t)(C::A_BASE + ai * A_COLS);
                    const uint64_t bd0 = bdesc_base + (uint64_t)((uint32_t)(bi * S::BSTAGE) >> 4);
                    const uint32_t first = ka == 0 ? 0u : 1u;    // accumulate unless first use of an accumulator
#pragma unroll
                    for (int half = 0; half < 2; ++half)
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
#pragma unroll
                            for (int op = 0; op < C::NOPS; ++op) {
                                const int mm = (half * 4 + kk) * C::NOPS + op;        // MMA index within the slab
                                const uint32_t boff = (uint32_t)(((half * C::NOPS + op) * S::REGION + kk * 32) >> 4);
                                ptx::mma_bf16_ts(dt0 + (uint32_t)((mm % C::NACC) * C::NMAX),
                                                 at0 + (uint32_t)((half * 4 + kk) * 8), bd0 + boff, idesc,
                                                 mm >= C::NACC ? 1u : first);
                            }
                    ptx::mma_commit(&b_empty[bi]);
                    ptx::mma_commit(&a_empty[ai]);
                }
                __syncwarp();
                issued = true;
                if (++bi == C::NB) { bi = 0; bph ^= 1u; }
                if (++ai == C::NA) { ai = 0; aph ^= 1u; }
            }
            if (!ok) break;
            if (ptx::elect_one()) ptx::mma_commit(&d_full[di]);
            __syncwarp();
            if (++di == 2) { di = 0; dph ^= 1u; }
        }
        if (!ok && lane == 0) fail();
        if (issued) {            // all MMAs retired before TMEM is released
            volatile int never = 0;
            if (ptx::elect_one()) ptx::mma_commit(mma_done);
            __syncwarp();
            __all_sync(0xFFFFFFFFu, ptx::mbar_wait(mma_done, 0, &never, LIM));
        }
    } else if (warp >= 8) {
        // ===================== converters: smem MXFP4 -> bf16 -> TMEM (A operand)
        const int cw = warp - 8, grp = cw >> 3, g = cw & 3, part = (cw >> 2) & 1;
        const int row = g * 32 + lane;
        const uint32_t t_lane = (uint32_t)(g * 32) << 16;
        const int my_tiles = (int)blockIdx.x < total ? (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
        const int n_slabs = my_tiles * slabs;
        static_assert(C::NW % C::GROUPS == 0 && C::NA % C::GROUPS == 0, "rings must split evenly between groups");
        bool ok = true;
        for (int i = grp; i < n_slabs; i += C::GROUPS) {
            const int wi = i % C::NW, ai = i % C::NA;
            const uint32_t wph = (uint32_t)((i / C::NW) & 1), aph = (uint32_t)((i / C::NA) & 1);
            if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&w_full[wi], wph, s_abort, LIM))) { ok = false; break; }
            const uint8_t *st = wring + wi * TILE_BYTES;
            const uint4 q0 = *reinterpret_cast<const uint4 *>(st + ((2 * part) * TILE_ROWS + row) * 16);
            const uint4 q1 = *reinterpret_cast<const uint4 *>(st + ((2 * part + 1) * TILE_ROWS + row) * 16);
            const uint32_t sc2 = *reinterpret_cast<const uint16_t *>(st + TILE_NIB_BYTES + row * 4 + 2 * part);
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&w_empty[wi]);
            const uint32_t s0 = sc2 & 0xFFu, s1 = sc2 >> 8;
            const bool big = __any_sync(0xFFFFFFFFu, s0 > 128u || s1 > 128u);
            uint32_t v[32];
            {
                const uint32_t m1 = scale_mult_lo(s0), m2 = scale_mult_hi(s0);
                decode_word(q0.x, m1, m2, big, v + 0);
                decode_word(q0.y, m1, m2, big, v + 4);
                decode_word(q0.z, m1, m2, big, v + 8);
                decode_word(q0.w, m1, m2, big, v + 12);
            }
            {
                const uint32_t m1 = scale_mult_lo(s1), m2 = scale_mult_hi(s1);
                decode_word(q1.x, m1, m2, big, v + 16);
                decode_word(q1.y, m1, m2, big, v + 20);
                decode_word(q1.z, m1, m2, big, v + 24);
                decode_word(q1.w, m1, m2, big, v + 28);
            }
            if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&a_empty[ai], aph ^ 1u, s_abort, LIM))) { ok = false; break; }
            ptx::tc_fence_after();
            ptx::tmem_st_32x32b_x32(tmem + t_lane + (uint32_t)(C::A_BASE + ai * A_COLS + part * 32), v);
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&a_full[ai]);
        }
        if (!ok && lane == 0) fail();
    } else if (warp < 4) {
        // ===================== epilogue: TMEM -> registers -> global
        const uint32_t t_lane = (uint32_t)(warp * 32) << 16;
        int di = 0;
        uint32_t dph = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
            Tile tl = decode_tile<C>(t, tile_start, E, MB, p.offsets, p.padded);
            if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&d_full[di], dph, s_abort, LIM))) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t dt = tmem + t_lane + (uint32_t)(di * C::D_COLS);
            for (int c0 = 0; c0 < tl.n; c0 += 16) {
                uint32_t raw[16];
                ptx::tmem_ld_32x32b_x16(dt + (uint32_t)c0, raw);
                ptx::tmem_wait_ld();
                for (int acc = 1; acc < nacc; ++acc) {          // sum the split accumulators
                    uint32_t part[16];
                    ptx::tmem_ld_32x32b_x16(dt + (uint32_t)(acc * C::NMAX + c0), part);
                    ptx::tmem_wait_ld();
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        raw[j] = __float_as_uint(__uint_as_float(raw[j]) + __uint_as_float(part[j]));
                }
                if (MODE == 0) {
                    // lane i < 16: gate of feature f; lane i + 16: up of the same f.
                    const bool is_gate = lane < 16;
                    const int f = tl.mb * 64 + warp * 16 + (lane & 15);
                    const float L = p.swiglu_limit;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const float send = __uint_as_float(is_gate ? raw[8 + j] : raw[j]);
                        const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, 16);
                        float gt = is_gate ? __uint_as_float(raw[j]) : recv;
                        float up = is_gate ? recv : __uint_as_float(raw[8 + j]);
                        if (L > 0.f) {
                            gt = fminf(gt, L);
                            up = fminf(fmaxf(up, -L), L);
                        }
                        const float h = silu_f(gt) * up;
                        const __nv_bfloat16 hh = __float2bfloat16_rn(h);
                        const __nv_bfloat16 hl = __float2bfloat16_rn(h - __bfloat162float(hh));
                        const int64_t r = (int64_t)tl.row0 + c0 + (is_gate ? j : 8 + j);
                        p.h_hi[r * p.I + f] = hh;
                        p.h_lo[r * p.I + f] = hl;
                    }
                } else {
                    const int c = tl.mb * TILE_ROWS + warp * 32 + lane;
                    const int my_pair = (lane < 16) ? __ldg(p.row_to_pair + tl.row0 + c0 + lane) : -1;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int pr = __shfl_sync(0xFFFFFFFFu, my_pair, j);
                        if (pr >= 0 && pr < p.P)
                            p.staging[(int64_t)pr * p.H + c] = __uint_as_float(raw[j]);
                        else if (pr >= p.P && lane == 0)
                            record_error(p.dev_error, DEV_ERR_ID_RANGE);
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&d_empty[di]);
            if (++di == 2) { di = 0; dph ^= 1u; }
        }
        if (!ok && lane == 0) fail();
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 5) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

// Gathered activations: row r of the permutation gets x[token(r)], padding
// rows (row_to_pair == -1) get zeros. Rows past padded[E] are not touched.
__global__ void gather_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ row_to_pair,
                              const int32_t *__restrict__ padded, int E, int H, int k, int64_t P,
                              uint16_t *__restrict__ xp, int32_t *dev_error)
{
    const int64_t R = __ldg(padded + E);
    const int vec = H / 8;
    for (int64_t r = blockIdx.x; r < R; r += gridDim.x) {
        const int32_t pr = __ldg(row_to_pair + r);
        uint4 *dst = reinterpret_cast<uint4 *>(xp + r * H);
        if (pr >= 0 && pr < P) {
            const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)(pr / k) * H);
            for (int v = threadIdx.x; v < vec; v += blockDim.x) dst[v] = __ldg(src + v);
        } else {
            if (pr >= P && threadIdx.x == 0) record_error(dev_error, DEV_ERR_ID_RANGE);
            for (int v = threadIdx.x; v < vec; v += blockDim.x) dst[v] = make_uint4(0, 0, 0, 0);
        }
    }
}

// y[t, c] = sum_j w[t, j] * staging[t*k + j, c], slots in ascending order.
__global__ void combine_kernel(const float *__restrict__ staging, const float *__restrict__ w, int T, int H,
                               int k, float *__restrict__ y)
{
    const int vec = H / 4;
    const int64_t n = (int64_t)T * vec;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / vec;
        const int c4 = (int)(i - t * vec);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j = 0; j < k; ++j) {
            const float wj = __ldg(w + t * k + j);
            const float4 s = __ldg(reinterpret_cast<const float4 *>(staging + (t * k + j) * H) + c4);
            acc.x = fmaf(wj, s.x, acc.x);
            acc.y = fmaf(wj, s.y, acc.y);
            acc.z = fmaf(wj, s.z, acc.z);
            acc.w = fmaf(wj, s.w, acc.w);
        }
        reinterpret_cast<float4 *>(y + t * H)[c4] = acc;
    }
}

template <class C>
cudaError_t launch_gemm(const GemmParams &p, int grid, cudaStream_t s)
{
    static unsigned long long attr_set = 0;   // bit d: attribute set on device d
    const size_t smem = Smem<C>::bytes(p.E);
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !((attr_set >> dev) & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)Smem<C>::bytes(1024));
        if (e != cudaSuccess) return e;
        if (dev < 64) __atomic_fetch_or(&attr_set, 1ull << dev, __ATOMIC_RELAXED);
    }
    moe_gemm_kernel<C><<<grid, C::THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

// Tile shape by the average rows per expert (T*k/E): decode batches get
// small tiles with deep pipelines, prefill batches large tiles.
enum class Regime { Tiny, Small, Mid, Large };

Regime pick_regime(int T, int k, int E)
{
    const double avg = (double)T * k / E;
    if (avg <= 2.0) return Regime::Tiny;
    if (avg <= 16.0) return Regime::Small;
    if (avg <= 64.0) return Regime::Mid;
    return Regime::Large;
}

}  // namespace

static void mark(const ForwardArgs &a, int i, cudaStream_t s)
{
    if (a.events && a.events[i]) cudaEventRecord(static_cast<cudaEvent_t>(a.events[i]), s);
}

cudaError_t launch_forward(const ForwardArgs &a, cudaStream_t s)
{
    const int64_t P = (int64_t)a.T * a.k;
    cudaError_t err;
    mark(a, 0, s);
    {
        int grid = (int)(a.rows_cap < 8192 ? a.rows_cap : 8192);
        gather_kernel<<<grid, 128, 0, s>>>(a.x, a.row_to_pair, a.padded, a.E, a.H, a.k, P, a.xp, a.dev_error);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    mark(a, 1, s);
    GemmParams g{};
    g.offsets = a.offsets;
    g.padded = a.padded;
    g.row_to_pair = a.row_to_pair;
    g.E = a.E;
    g.I = a.I;
    g.H = a.H;
    g.k = a.k;
    g.swiglu_limit = a.swiglu_limit;
    g.P = P;
    g.h_hi = reinterpret_cast<__nv_bfloat16 *>(a.h_hi);
    g.h_lo = reinterpret_cast<__nv_bfloat16 *>(a.h_lo);
    g.staging = a.staging;
    g.dev_error = a.dev_error;

    // W13: K = H, 64 features (128 rows) per weight tile
    g.tm_b0 = *a.tmap_xp;
    g.tm_b1 = *a.tmap_xp;
    g.wpack = a.packed;
    g.K = a.H;
    g.MB = a.I / 64;
    const Regime rg = pick_regime(a.T, a.k, a.E);
    err = rg == Regime::Tiny  ? launch_gemm<W13Tiny>(g, a.num_sms, s)
        : rg == Regime::Small ? launch_gemm<W13Small>(g, a.num_sms, s)
        : rg == Regime::Mid   ? launch_gemm<W13Mid>(g, a.num_sms, s)
                              : launch_gemm<W13Large>(g, a.num_sms, s);
    if (err != cudaSuccess) return err;
    mark(a, 2, s);

    // W2: K = I, 128 output features per weight tile
    g.tm_b0 = *a.tmap_hhi;
    g.tm_b1 = *a.tmap_hlo;
    g.wpack = a.packed + packed_w13_bytes(a.E, a.H, a.I);
    g.K = a.I;
    g.MB = a.H / TILE_ROWS;
    err = rg == Regime::Tiny  ? launch_gemm<W2Tiny>(g, a.num_sms, s)
        : rg == Regime::Small ? launch_gemm<W2Small>(g, a.num_sms, s)
        : rg == Regime::Mid   ? launch_gemm<W2Mid>(g, a.num_sms, s)
                              : launch_gemm<W2Large>(g, a.num_sms, s);
    if (err != cudaSuccess) return err;
    mark(a, 3, s);

    {
        const int64_t n = (int64_t)a.T * (a.H / 4);
        int grid = (int)((n + 255) / 256);
        if (grid > 4 * 1024) grid = 4 * 1024;
        if (grid < 1) grid = 1;
        combine_kernel<<<grid, 256, 0, s>>>(a.staging, a.topk_w, a.T, a.H, a.k, a.y);
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    mark(a, 4, s);
    note_launch(4);
    return cudaSuccess;
}

}  // namespace moe

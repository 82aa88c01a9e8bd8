// Decode layer GEMMs in one persistent launch: W13 (+ SiLU*up + h terms) and W2
// over one tile list, for batches of at most 2 rows per expert (sm_103a).
//
// Method: "DeepSeek V4 Flash 单卡 MI300X" (txtmix.com) §三 — grouped MXFP4
// expert GEMMs with SiLU(gate)*up fused into the W13 epilogue, then W2; §九 —
// the optional SwiGLU clamp. Same tiles and arithmetic as the 16-row
// weight-major tiles of gemm.cu (swap-AB: 128 weight rows x 16 token rows x 2
// MXFP8 terms, two-slab stages, two MMA warps; with at most 8 tokens, 8 token
// rows and a sixth weight stage); see there for the operand and scale-factor
// layouts.
//
// What the single launch adds: a CTA walks the W13 tiles of the tile list and
// then the W2 tiles, all in the same rings. A W2 tile of expert e may start as
// soon as every W13 tile of e has stored its h rows: each W13 tile's
// epilogue, after its h stores, makes them visible to the async proxy that
// the TMA copies of h go through (fence.proxy.async) and device-wide, and adds
// one to e's counter (release);
// the activation producer of a W2 tile of e waits (acquire, bounded) for the
// counter to reach e's W13 tile count before its first copy of h. W13 tiles
// never wait on anything of W2, so no wait is circular, and the tile list is
// expert-major, so the W2 tiles a CTA meets first belong to experts whose W13
// tiles finished long before. With two launches, an SM whose last W13 tile
// ended early idled until the last SM's did; here it goes on with W2 tiles
// and their weight stream. The counters live in the workspace; the gather
// zeroes them.
//
// Both GEMMs need an even number of 128-K slabs per tile (H and I multiples of
// 256) and at least two stages per tile (H, I >= 512), so a stage never spans
// two tiles and both MMA warps write every tile.
// Warp roles (384 threads): 0-3 epilogue, 4-7 scale-factor copiers, 8 and 11
// MMA issuers, 9 activation producer, 10 weight producer. Every wait is
// bounded (2 s); on time-out a CTA records MOE_ERR_TIMEOUT, drains its copies
// and MMAs, frees TMEM and exits.
#include <cuda_bf16.h>

#include <cstdint>

#include "gemm_common.cuh"
#include "moe_internal.h"
#include "mxfp4_tile.cuh"
#include "mxfp8_terms.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

// NMAX token rows per tile: 16, or 8 when no expert can hold more (at most 8 tokens), which halves
// the activation stages and leaves room for a sixth weight stage.
template <int NMAX_>
struct DCfg {
    static constexpr int NMAX = NMAX_, NT = 2, NP = NT * NMAX;   // token rows per tile, terms, MMA N
    static constexpr int SPS = 2;                                 // slabs per stage
    static constexpr int NA = NMAX == 8 ? 6 : 5, NB = 4, NSF = 6, MW = 2, ND = 8, EMAX = 512;
    static constexpr int SF_COLS = 8;                          // one slab's cell: A (4 columns), B (1), pad
    static constexpr int CELL_COLS = SPS * SF_COLS;
    static constexpr int D_COLS = NP;                          // one accumulator set
    static constexpr int SF_BASE = 2 * MW * D_COLS;            // [MMA warp][double buffer]
    static constexpr int THREADS = 384;
    static_assert(SF_BASE + NSF * CELL_COLS <= TMEM_COLS, "TMEM budget");
    static_assert(NA <= ND && NB <= ND && NSF <= ND, "done ring");
};

template <class C>
struct DSmem {
    static constexpr int ASTAGE = C::SPS * SLAB_SMEM_BYTES;   // expanded E2M1 slabs
    static constexpr int BSLAB = C::NP * 128;                 // [term][row][128 K bytes]
    static constexpr int BSTAGE = C::SPS * BSLAB;
    static constexpr int BSSLAB = C::NP * 4;                  // scale words [term][row] of one slab
    static constexpr int BSSTAGE = (C::SPS * BSSLAB + 127) / 128 * 128;
    static constexpr int SFSTAGE = C::SPS * SLAB_SF_BYTES;
    static constexpr int A_OFF = 0;
    static constexpr int B_OFF = A_OFF + C::NA * ASTAGE;
    static constexpr int SF_OFF = B_OFF + C::NB * BSTAGE;
    static constexpr int BS_OFF = SF_OFF + C::NA * SFSTAGE;
    static constexpr int BAR_OFF = BS_OFF + C::NB * BSSTAGE;
    static constexpr int NBARS = C::NA + C::NB + C::NSF + C::ND + 2 * 2 + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int PAIRMAX_OFF = MISC_OFF + 16;         // W13 epilogue: [2 buffers][4 warps][16] floats
    static constexpr int PREFIX_OFF = PAIRMAX_OFF + 2 * 4 * 16 * 4;
    // W13 and W2 tile prefixes [E + 1] each, scan scratch [32], first padded row and row count [E] each
    static constexpr size_t bytes(int E) { return 1024 + PREFIX_OFF + sizeof(int) * (size_t)(4 * E + 2 + 32); }
    static_assert(BSLAB % 1024 == 0 && ASTAGE % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
};
static_assert(DSmem<DCfg<16>>::bytes(DCfg<16>::EMAX) <= 232448, "shared memory per CTA");
static_assert(DSmem<DCfg<8>>::bytes(DCfg<8>::EMAX) <= 232448, "shared memory per CTA");

struct DecodeParams {
    GemmParams g13, g2;    // W13 (x terms in, h terms out) and W2 (h terms in, staging or y out)
    uint32_t *done13;      // [E]: W13 tiles of each expert whose h rows are stored
};

// tile t of the combined list -> (GEMM, tile of that GEMM)
struct DTile {
    int w2;      // 0: W13, 1: W2
    Tile t;
};

template <class C, bool FAST>
__global__ void __launch_bounds__(C::THREADS, 1) moe_gemm_decode_kernel(const __grid_constant__ DecodeParams dp)
{
    using S = DSmem<C>;
    constexpr int NMAX = C::NMAX, NT = C::NT, NP = C::NP, SPS = C::SPS;
    const GemmParams &p13 = dp.g13;
    const GemmParams &p2 = dp.g2;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *aring = smem + S::A_OFF;
    uint8_t *bring = smem + S::B_OFF;
    uint8_t *sfring = smem + S::SF_OFF;
    uint8_t *bsring = smem + S::BS_OFF;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S::BAR_OFF);
    uint64_t *a_full = bars, *b_full = a_full + C::NA, *sf_full = b_full + C::NB;
    uint64_t *done = sf_full + C::NSF;
    uint64_t *d_full = done + C::ND, *d_empty = d_full + 2;
    uint64_t *mma_done = d_empty + 2;
    uint32_t *s_tmem = reinterpret_cast<uint32_t *>(smem + S::MISC_OFF);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + S::MISC_OFF + 4);
    float *pairmax = reinterpret_cast<float *>(smem + S::PAIRMAX_OFF);
    const int E = p13.E;
    int *ts13 = reinterpret_cast<int *>(smem + S::PREFIX_OFF);   // [E + 1]
    int *ts2 = ts13 + E + 1;                                      // [E + 1]
    int *scan_tmp = ts2 + E + 1;                                  // [32]
    int *s_pad0 = scan_tmp + 32, *s_cnt = s_pad0 + E;             // [E] each

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int MB13 = p13.MB, MB2 = p2.MB;
    const int slabs13 = p13.K / KSLAB, slabs2 = p2.K / KSLAB;

    // ---- tile prefixes over experts, W13 and W2 (E <= 512: two experts per thread)
    {
        int v13[2], v2[2];
        int s13 = 0, s2 = 0;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const int e = tid * 2 + q;
            const int cnt = e < E ? (__ldg(p13.offsets + e + 1) - __ldg(p13.offsets + e)) : 0;
            if (e < E) {
                s_cnt[e] = cnt;
                s_pad0[e] = __ldg(p13.padded + e);
            }
            const int blocks = (cnt + NMAX - 1) / NMAX;
            v13[q] = blocks * MB13;
            v2[q] = blocks * MB2;
            s13 += v13[q];
            s2 += v2[q];
        }
        // two block scans: the W13 prefix, then the W2 prefix
        for (int which = 0; which < 2; ++which) {
            const int s = which ? s2 : s13;
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
            int *ts = which ? ts2 : ts13;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int e = tid * 2 + q;
                if (e < E) ts[e] = run;
                run += which ? v2[q] : v13[q];
            }
            if (tid == C::THREADS - 1) ts[E] = run;
            __syncthreads();
        }
    }
    const int total13 = ts13[E], total = total13 + ts2[E];
    if ((int)blockIdx.x >= total) {           // uniform: this CTA has no tiles
        griddep_wait();
        return;
    }

    // ---- barriers and TMEM
    if (tid == 0) {
        for (int i = 0; i < C::NA; ++i) ptx::mbar_init(&a_full[i], 1);
        for (int i = 0; i < C::NB; ++i) ptx::mbar_init(&b_full[i], 1);
        for (int i = 0; i < C::NSF; ++i) ptx::mbar_init(&sf_full[i], 4);
        for (int i = 0; i < C::ND; ++i) ptx::mbar_init(&done[i], 1);
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&d_full[i], C::MW);    // one commit per MMA warp and tile
            ptx::mbar_init(&d_empty[i], 4);
        }
        ptx::mbar_init(mma_done, C::MW);
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
    const int my_tiles = (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1;
    const uint64_t LIM = WAIT_LIMIT_NS;

    auto fail = [&]() {
        *s_abort = 1;
        record_error(p13.dev_error, DEV_ERR_TIMEOUT);
    };
    auto wait_done = [&](int q) -> bool {
        return q < 0 || ptx::mbar_wait(&done[q % C::ND], (uint32_t)((q / C::ND) & 1), s_abort, LIM);
    };
    auto tile_of = [&](int j) -> DTile {
        const int t = (int)blockIdx.x + j * (int)gridDim.x;
        DTile d;
        d.w2 = t >= total13;
        d.t = d.w2 ? decode_tile<NMAX>(t - total13, ts2, E, MB2, s_cnt, s_pad0)
                   : decode_tile<NMAX>(t, ts13, E, MB13, s_cnt, s_pad0);
        return d;
    };
    auto stages_of = [&](const DTile &d) { return (d.w2 ? slabs2 : slabs13) / SPS; };

    if (warp == 10) {
        // ===================== weight producer: per stage one TMA box of two slabs (E2M1 rows, expanded in
        // shared memory) and one bulk copy of their scales
        if (ptx::elect_one()) {
            ptx::prefetch_tmap(&p13.tm_a);
            ptx::prefetch_tmap(&p2.tm_a);
        }
        __syncwarp();
        int ai = 0, s = 0;
        long long issued = 0;
        bool ok = true;
        for (int j = 0; j < my_tiles && ok; ++j) {
            const DTile d = tile_of(j);
            const GemmParams &g = d.w2 ? p2 : p13;
            const int slabs = d.w2 ? slabs2 : slabs13;
            for (int st = 0; st < slabs / SPS; ++st, ++s) {
                if (!__all_sync(0xFFFFFFFFu, wait_done(s - C::NA))) { ok = false; break; }
                if (ptx::elect_one()) {
                    const int r0 = ((d.t.e * g.MB + d.t.mb) * slabs + st * SPS) * TILE_ROWS;
                    ptx::mbar_arrive_expect_tx(&a_full[ai], (uint32_t)(SPS * (SLAB_NIB_BYTES + SLAB_SF_BYTES)));
                    ptx::tma_load_2d(aring + ai * S::ASTAGE, &g.tm_a, 0, r0, &a_full[ai]);
                    ptx::bulk_g2s(sfring + ai * S::SFSTAGE, g.wsf + (size_t)(r0 / TILE_ROWS) * SLAB_SF_BYTES,
                                  (uint32_t)(SPS * SLAB_SF_BYTES), &a_full[ai]);
                }
                __syncwarp();
                ++issued;
                if (++ai == C::NA) ai = 0;
            }
        }
        if (!ok && lane == 0) fail();
        volatile int never = 0;
        for (long long i = 1; i <= (issued < C::NA ? issued : C::NA); ++i) {
            const long long n = issued - i;
            __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&a_full[n % C::NA], (uint32_t)((n / C::NA) & 1), &never, LIM));
        }
    } else if (warp == 9) {
        // ===================== activation producer: per stage one 4-D TMA box of the terms (128 K x 16 rows x
        // 2 terms x 2 slabs) and one 3-D box of their scale words. x comes from the gather (the kernel
        // before); h of a W2 tile from this grid's W13 tiles of the same expert (counter wait).
        if (ptx::elect_one()) {
            ptx::prefetch_tmap(&p13.tm_b);
            ptx::prefetch_tmap(&p13.tm_bs);
            ptx::prefetch_tmap(&p2.tm_b);
            ptx::prefetch_tmap(&p2.tm_bs);
        }
        griddep_wait();
        if (lane == 0) griddep_launch_dependents();
        __syncwarp();
        int bi = 0, s = 0;
        long long issued = 0;
        bool ok = true;
        for (int j = 0; j < my_tiles && ok; ++j) {
            const DTile d = tile_of(j);
            const GemmParams &g = d.w2 ? p2 : p13;
            if (d.w2) {
                // every W13 tile of this expert must have stored its h rows
                // (every lane acquires, so the copies below are ordered after it whichever lane issues them)
                const uint32_t need = (uint32_t)(ts13[d.t.e + 1] - ts13[d.t.e]);
                const uint64_t t0 = ptx::globaltimer_ns();
                bool got = true;
                while (!__all_sync(0xFFFFFFFFu, ptx::ld_acquire_gpu(dp.done13 + d.t.e) >= need)) {
                    if (__any_sync(0xFFFFFFFFu, *s_abort != 0 || ptx::globaltimer_ns() - t0 > LIM)) { got = false; break; }
                    ptx::nanosleep_ns(200);
                }
                ptx::fence_proxy_async_global();       // the copies below read what the acquire made visible
                if (!got) { ok = false; break; }
            }
            const int slabs = d.w2 ? slabs2 : slabs13;
            for (int st = 0; st < slabs / SPS; ++st, ++s) {
                if (!__all_sync(0xFFFFFFFFu, wait_done(s - C::NB))) { ok = false; break; }
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(&b_full[bi], (uint32_t)(SPS * (S::BSLAB + S::BSSLAB)));
                    ptx::tma_load_4d(bring + bi * S::BSTAGE, &g.tm_b, 0, d.t.row0, 0, st * SPS, &b_full[bi]);
                    ptx::tma_load_3d(bsring + bi * S::BSSTAGE, &g.tm_bs, d.t.row0, 0, st * SPS, &b_full[bi]);
                }
                __syncwarp();
                ++issued;
                if (++bi == C::NB) bi = 0;
            }
        }
        if (!ok && lane == 0) fail();
        volatile int never = 0;
        for (long long i = 1; i <= (issued < C::NB ? issued : C::NB); ++i) {
            const long long n = issued - i;
            __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&b_full[n % C::NB], (uint32_t)((n / C::NB) & 1), &never, LIM));
        }
    } else if (warp >= 4 && warp < 8) {
        // ===================== scale-factor copiers: per stage and slab, A's 4 columns (weight stage) and B's
        // word per B row (activation stage) into the next TMEM cell of this warp's lane quarter
        int ai = 0, bi = 0, sc = 0, s = 0;
        uint32_t aph = 0, bph = 0;
        bool ok = true;
        const uint32_t quarter = (uint32_t)((warp & 3) * 32) << 16;
        for (int j = 0; j < my_tiles && ok; ++j) {
            const int nst = stages_of(tile_of(j));
            for (int st = 0; st < nst; ++st, ++s) {
                if (!__all_sync(0xFFFFFFFFu, wait_done(s - C::NSF) && ptx::mbar_wait(&a_full[ai], aph, s_abort, LIM) &&
                                                 ptx::mbar_wait(&b_full[bi], bph, s_abort, LIM))) { ok = false; break; }
                ptx::tc_fence_after();
#pragma unroll
                for (int pos = 0; pos < SPS; ++pos) {
                    const uint4 aw = *reinterpret_cast<const uint4 *>(sfring + ai * S::SFSTAGE + pos * SLAB_SF_BYTES + lane * 16);
                    const uint32_t *bs = reinterpret_cast<const uint32_t *>(bsring + bi * S::BSSTAGE + pos * S::BSSLAB);
                    const uint32_t bw = lane < NP ? bs[lane] : 0u;                          // B row j = lane
                    const uint32_t v8[8] = {aw.x, aw.y, aw.z, aw.w, bw, 0u, 0u, 0u};
                    ptx::tmem_st_32x32b_x8(tmem + quarter + (uint32_t)(C::SF_BASE + sc * C::CELL_COLS + pos * C::SF_COLS), v8);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(&sf_full[sc]);
                if (++ai == C::NA) { ai = 0; aph ^= 1u; }
                if (++bi == C::NB) { bi = 0; bph ^= 1u; }
                if (++sc == C::NSF) sc = 0;
            }
        }
        if (!ok && lane == 0) fail();
    } else if (warp == 8 || warp == 11) {
        // ===================== MMA issuers: the tile's stage st belongs to warp st % 2 and its own accumulator set; both
        // warps walk every stage and commit every tile, so the epilogue sees one arrival per warp and tile
        const int q = warp == 8 ? 0 : 1;
        const uint64_t adesc0 = ptx::smem_desc_sw128(ptx::smem_u32(aring));
        const uint64_t bdesc0 = ptx::smem_desc_sw128(ptx::smem_u32(bring));
        int ai = 0, bi = 0, sc = 0, di = 0, s = 0;
        uint32_t sph = 0, dph = 0;
        bool ok = true;
        for (int j = 0; j < my_tiles && ok; ++j) {
            const int nst = stages_of(tile_of(j));
            if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&d_empty[di], dph ^ 1u, s_abort, LIM))) { ok = false; break; }
            ptx::tc_fence_after();
            int mine_in_tile = 0;          // this warp's 32-K blocks in the tile so far
            for (int st = 0; st < nst; ++st, ++s) {
                const bool mine = (st % C::MW) == q;     // counted from the tile's start, as in gemm.cu
                if (mine) {
                    if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&sf_full[sc], sph, s_abort, LIM))) { ok = false; break; }
                    ptx::tc_fence_after();
                }
                const bool tile_end = st == nst - 1;
                if (mine || tile_end) {
                    if (ptx::elect_one()) {
                        if (mine) {
                            const uint32_t dt = tmem + (uint32_t)((q * 2 + di) * C::D_COLS);
#pragma unroll
                            for (int pos = 0; pos < SPS; ++pos) {
                                const uint64_t ad = adesc0 + (uint64_t)((uint32_t)(ai * S::ASTAGE + pos * SLAB_SMEM_BYTES) >> 4);
                                const uint64_t bd = bdesc0 + (uint64_t)((uint32_t)(bi * S::BSTAGE + pos * S::BSLAB) >> 4);
                                const uint32_t sfa = tmem + (uint32_t)(C::SF_BASE + sc * C::CELL_COLS + pos * C::SF_COLS);
#pragma unroll
                                for (int kb = 0; kb < 4; ++kb) {
                                    const int kk = mine_in_tile + 4 * pos + kb;    // overwrite on the warp's first
                                    ptx::mma_mx_ss(dt, ad + (uint64_t)(kb * 2), bd + (uint64_t)(kb * 2),
                                                   ptx::idesc_mx_e2m1_e4m3(128, NP, (uint32_t)kb), sfa, sfa + 4,
                                                   kk > 0 ? 1u : 0u);
                                }
                            }
                            ptx::mma_commit(&done[s % C::ND]);
                        }
                        if (tile_end) ptx::mma_commit(&d_full[di]);
                    }
                    __syncwarp();
                }
                if (mine) mine_in_tile += 4 * SPS;
                if (++ai == C::NA) ai = 0;
                if (++bi == C::NB) bi = 0;
                if (++sc == C::NSF) { sc = 0; sph ^= 1u; }
            }
            if (++di == 2) { di = 0; dph ^= 1u; }
        }
        if (!ok && lane == 0) fail();
        volatile int never = 0;
        if (ptx::elect_one()) ptx::mma_commit(mma_done);
        __syncwarp();
        if (q == 0) __all_sync(0xFFFFFFFFu, ptx::mbar_wait(mma_done, 0, &never, LIM));
    } else if (warp < 4) {
        // ===================== epilogue: TMEM -> registers -> global, one chunk of NMAX columns per term and
        // tile. W13 tiles pair warps at named barriers (1 and 2) and meet all four
        // epilogue warps at barrier 3 before publishing the tile, so no warp leaves the loop early: after
        // a failed wait a warp skips the work but still meets the others at every barrier.
        const uint32_t t_lane = (uint32_t)(warp * 32) << 16;
        int di = 0, chunk = 0;
        uint32_t dph = 0;
        bool ok = true;
        for (int j = 0; j < my_tiles; ++j) {
            const DTile d = tile_of(j);
            const Tile &tl = d.t;
            ok = ok && __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&d_full[di], dph, s_abort, LIM));
            ptx::tc_fence_after();
            constexpr int HALF = NMAX / 2;
            uint32_t raw[NMAX];
#pragma unroll
            for (int q = 0; q < NMAX; ++q) raw[q] = 0u;
            if (ok) {
                // both MMA warps wrote every tile: sum their sets' term columns (term t, token q at column
                // t * NMAX + q of the set) in (warp, term) order
                uint32_t part[C::MW][C::D_COLS];
#pragma unroll
                for (int w = 0; w < C::MW; ++w)
#pragma unroll
                    for (int c = 0; c < C::D_COLS; c += 16)
                        ptx::tmem_ld_32x32b_x16(tmem + t_lane + (uint32_t)((w * 2 + di) * C::D_COLS + c),
                                                *reinterpret_cast<uint32_t (*)[16]>(&part[w][c]));
                ptx::tmem_wait_ld();
#pragma unroll
                for (int u = 0; u < C::MW * NT; ++u)
#pragma unroll
                    for (int q = 0; q < NMAX; ++q)
                        raw[q] = __float_as_uint(__uint_as_float(raw[q]) + __uint_as_float(part[u / NT][(u % NT) * NMAX + q]));
            }
            if (!d.w2) {
                const GemmParams &g = p13;
                // lane i < 16: gate of feature f; lane i + 16: up of the same f. Lane i ends with h[f] for
                // tokens 0 .. HALF-1 of the tile, lane i + 16 for tokens HALF .. NMAX-1.
                const bool is_gate = lane < 16;
                const int f = tl.mb * 64 + warp * 16 + (lane & 15);
                const float L = g.swiglu_limit;
                float h[HALF], am[HALF];
#pragma unroll
                for (int q = 0; q < HALF; ++q) {
                    const float send = __uint_as_float(is_gate ? raw[HALF + q] : raw[q]);
                    const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, 16);
                    float gt = is_gate ? __uint_as_float(raw[q]) : recv;
                    float up = is_gate ? recv : __uint_as_float(raw[HALF + q]);
                    if (L > 0.f) {
                        gt = fminf(gt, L);
                        up = fminf(fmaxf(up, -L), L);
                    }
                    h[q] = silu_f(gt) * up;
                    am[q] = fabsf(h[q]);
                }
                // W2 scale blocks are 32 consecutive features: 16 in this half-warp, 16 in the partner warp
                // (warps 0+1 and 2+3), which trade maxima through shared memory
#pragma unroll
                for (int q = 0; q < HALF; ++q)
#pragma unroll
                    for (int o = 1; o < 16; o <<= 1) am[q] = fmaxf(am[q], __shfl_xor_sync(0xFFFFFFFFu, am[q], o));
                float *pm = pairmax + (chunk & 1) * 64;
                if ((lane & 15) == 0)
#pragma unroll
                    for (int q = 0; q < HALF; ++q) pm[warp * 16 + (lane >> 4) * HALF + q] = am[q];
                ptx::bar_sync_n(1 + (warp >> 1), 64);
                if (ok) {
                    const int blk = f >> 5;                      // W2 K-block of this feature
                    const bool writes_scale = (lane & 15) == 0 && (warp & 1) == 0;
#pragma unroll
                    for (int q = 0; q < HALF; q += 2) {        // two token rows per conversion
                        const float *pmq = pm + (warp ^ 1) * 16 + (lane >> 4) * HALF + q;
                        const int e0 = mxfp8_block_exp(fmaxf(am[q], pmq[0]));
                        const int e1 = mxfp8_block_exp(fmaxf(am[q + 1], pmq[1]));
                        const int64_t row = (int64_t)tl.row0 + (lane >> 4) * HALF + q;
                        float r0 = h[q], r1 = h[q + 1];
#pragma unroll
                        for (int term = 0; term < NT; ++term) {
                            uint32_t sb0, sb1;
                            const uint32_t v = mxfp8_term_2x(r0, r1, e0, e1, term, sb0, sb1);
                            uint8_t *dq = g.hq + (((int64_t)(f >> 7) * NT + term) * g.rows_cap + row) * 128 + (f & 127);
                            dq[0] = (uint8_t)v;
                            dq[128] = (uint8_t)(v >> 8);
                            if (writes_scale) {
                                uint8_t *ds = g.hs + (((int64_t)(blk >> 2) * NT + term) * g.rows_sf + row) * 4 + (blk & 3);
                                ds[0] = (uint8_t)sb0;
                                ds[4] = (uint8_t)sb1;
                            }
                        }
                    }
                }
                // publish the tile's h rows: visible to the async proxy and device-wide, then one release add
                ptx::fence_proxy_async_global();
                __threadfence();
                ptx::bar_sync_n(3, 128);
                if (ok && warp == 0 && lane == 0) ptx::red_release_gpu_add(dp.done13 + tl.e, 1u);
                ++chunk;
            } else if (ok) {
                const GemmParams &g = p2;
                const int c = tl.mb * TILE_ROWS + warp * 32 + lane;
                const int my_pair = (lane < NMAX) ? __ldg(g.row_to_pair + tl.row0 + lane) : -1;
                if constexpr (FAST) {
                    // fast combine: w * o added into the token's row of y; lane q < NMAX holds row q's weight
                    const float my_w = (my_pair >= 0 && my_pair < g.P) ? __ldg(g.topk_w + my_pair) : 0.f;
#pragma unroll
                    for (int q = 0; q < NMAX; ++q) {
                        const int pr = __shfl_sync(0xFFFFFFFFu, my_pair, q);
                        const float wq = __shfl_sync(0xFFFFFFFFu, my_w, q);
                        if (pr >= 0 && pr < g.P)
                            ptx::red_add_f32(g.y + (int64_t)(pr / g.k) * g.H + c, wq * __uint_as_float(raw[q]));
                        else if (pr >= g.P && lane == 0)
                            record_error(g.dev_error, DEV_ERR_ID_RANGE);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < NMAX; ++q) {
                        const int pr = __shfl_sync(0xFFFFFFFFu, my_pair, q);
                        if (pr >= 0 && pr < g.P)
                            g.staging[(int64_t)pr * g.H + c] = __uint_as_float(raw[q]);
                        else if (pr >= g.P && lane == 0)
                            record_error(g.dev_error, DEV_ERR_ID_RANGE);
                    }
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (ok && lane == 0) ptx::mbar_arrive(&d_empty[di]);
            if (++di == 2) { di = 0; dph ^= 1u; }
        }
        if (!ok && lane == 0) fail();
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    if (warp == 8) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

template <class C, bool FAST>
cudaError_t launch_decode(const DecodeParams &p, int grid, cudaStream_t s, bool pdl)
{
    static unsigned long long attr_set = 0;   // bit d: attribute set on device d
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !((attr_set >> dev) & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(moe_gemm_decode_kernel<C, FAST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)DSmem<C>::bytes(C::EMAX));
        if (e != cudaSuccess) return e;
        if (dev < 64) __atomic_fetch_or(&attr_set, 1ull << dev, __ATOMIC_RELAXED);
    }
    return launch_ex(moe_gemm_decode_kernel<C, FAST>, dim3(grid), dim3(C::THREADS), DSmem<C>::bytes(p.g13.E), s, pdl, p);
}

}  // namespace

bool decode_fused_supported(int H, int I, int E)
{
    return E <= DCfg<16>::EMAX && H % 256 == 0 && I % 256 == 0 && H >= 512 && I >= 512;
}

cudaError_t launch_gemm_decode(const GemmParams &g13, const GemmParams &g2, uint32_t *done13, bool fast, bool rows8,
                               int grid, cudaStream_t s, bool pdl)
{
    DecodeParams p;
    p.g13 = g13;
    p.g2 = g2;
    p.done13 = done13;
    if (rows8) return fast ? launch_decode<DCfg<8>, true>(p, grid, s, pdl) : launch_decode<DCfg<8>, false>(p, grid, s, pdl);
    return fast ? launch_decode<DCfg<16>, true>(p, grid, s, pdl) : launch_decode<DCfg<16>, false>(p, grid, s, pdl);
}

}  // namespace moe

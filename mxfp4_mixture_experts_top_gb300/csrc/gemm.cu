// Grouped MXFP4 expert GEMMs on tcgen05 block-scaled MMAs (sm_103a), plus the
// gather that turns activations into MXFP8 terms and the routing-weighted
// combine.
//
// Method: "DeepSeek V4 Flash 单卡 MI300X" (txtmix.com) §三 — grouped MXFP4
// expert GEMMs, W13 with SiLU(gate)*up fused into its epilogue over a gate/up
// interleaved weight layout, then W2; §九 — the optional SwiGLU clamp. The
// combine y[t] = sum_j w[t,j] o_j is the routing-weighted scatter back to
// token order.
//
// Design (swap-AB: weights are the M = 128 side, token rows the N side):
//   * A = 128 weight rows x K as E2M1, fetched by TMA straight from the
//     prepacked HBM layout into the padded shared-memory operand layout of
//     tcgen05 kind::mxf8f6f4; A's E8M0 scales ride in the same stage and four
//     warps copy them into a tensor-memory ring of scale-factor cells. No
//     instruction of the SM decodes a weight: the tensor core applies the
//     scales (block_scale, one scale per 32 K-elements, K = 32 per MMA).
//   * B = the tile's token rows as NT MXFP8 terms (x: 2 terms, h: 2; see
//     mxfp8_terms.cuh), stacked along N: B row t * NMAX + n is term t of token
//     row n, so one MMA per 32-K block covers all terms and reads A once.
//   * D = fp32 accumulators in TMEM, double-buffered so the epilogue of one
//     tile overlaps the main loop of the next; the epilogue adds the NT term
//     columns and the NACC accumulators of each token.
//   * Persistent CTAs (one per SM) walk a tile list built on the device from
//     the permutation offsets: expert-major, then token block, then weight
//     row tile, so concurrent CTAs share B tiles in L2.
//   * W13's epilogue applies SiLU(gate)*up, then splits h into two MXFP8 terms
//     for W2 (block maxima over 32 features span two epilogue warps, which
//     exchange them through shared memory).
//   * Per stage the MMA issuer waits on one barrier (the stage's scale-factor
//     cell, filled after its weights and activations landed) and makes one
//     commit, to done[s % ND], which frees the stage in all rings at once.
//   * Under programmatic dependent launch the prologue and the weight stream
//     run while the previous kernel finishes; only the activation producer
//     waits for it (griddepcontrol.wait).
// Warp roles (352 threads, 384 with the second MMA issuer): 0-3 epilogue, 4-7
// scale-factor copiers (one per TMEM lane quarter: the tensor core's
// sub-partition q reads the scale factors of its 32 A rows, and of every B
// row, from lane quarter q, so each quarter holds a full copy), 8 MMA issuer
// and TMEM owner, 9 activation producer (4-D TMA of the terms, 3-D TMA of
// their scale words), 10 weight producer (2-D TMA + bulk copy of the scales),
// 11 second MMA issuer (decode configurations).
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

// Kernel configuration. MODE 0: W13 (x terms -> SiLU(gate)*up -> h terms),
// MODE 1: W2 (h terms -> per-pair outputs). NMAX: most token rows per tile
// (experts with more rows get several tiles). NT: activation terms. SPS:
// K-slabs per ring stage. Every ring (weights, activations with their scales,
// TMEM scale-factor cells) advances one stage per producer / copier / MMA
// step, so each step's fixed cost (barrier waits and arrivals, copy issue: a
// few hundred cycles) is paid once per SPS slabs. NA / NB: weight /
// activation ring stages. NSF: TMEM scale-factor cells (one stage each).
// NACC: accumulators per tile and MMA warp (consecutive 32-K blocks rotate
// over them, so short MMAs do not wait on each other). MW: MMA warps; stage s
// is issued by warp s % MW into its own accumulator sets, so while one warp
// waits and does its bookkeeping the other keeps the tensor pipe fed. EMAX: most experts the
// configuration takes (its shared memory holds per-expert tile prefixes, first rows and counts).
// NTO: MXFP8 terms of h the W13 epilogue writes (MODE 0; the NT of the matching W2 configuration).
template <int MODE_, int NMAX_, int NT_, int SPS_, int NA_, int NB_, int NSF_, int NACC_, int MW_, int EMAX_ = 1024,
          int NTO_ = 3>
struct Cfg {
    static constexpr int MODE = MODE_, NMAX = NMAX_, NT = NT_, SPS = SPS_, NA = NA_, NB = NB_, NSF = NSF_,
                         NACC = NACC_, MW = MW_, EMAX = EMAX_, NTO = NTO_;
    static constexpr int NP = NT * NMAX;                       // MMA N: all terms of NMAX rows
    static constexpr int SFB_COLS = (NP + 31) / 32;            // B scale cells: row j in column j / 32
    static constexpr int SF_COLS = (4 + SFB_COLS + 3) / 4 * 4; // one slab's cells: A (4 columns), then B
    static constexpr int CELL_COLS = SPS * SF_COLS;            // one stage
    static constexpr int D_COLS = NACC * NP;                   // one accumulator set
    static constexpr int SF_BASE = 2 * MW * D_COLS;            // [MMA warp][double buffer][set]
    static constexpr int THREADS = 352 + 32 * (MW - 1);
    // Stage s's MMAs complete -> done[s % ND]: frees the stage in the weight, activation and scale-factor
    // rings at once. A waiter for stage s - N (N = NA, NB or NSF) cannot see the barrier a full lap
    // ahead, since that needs stage s - N + ND >= s, which it has not filled yet.
    static constexpr int ND = 8;
    static_assert(NA <= ND && NB <= ND && NSF <= ND, "done ring");
    static_assert(NP % 16 == 0 && NP <= 256, "MMA N");
    static_assert(NMAX % 16 == 0, "token rows per tile");
    static_assert(SF_BASE + NSF * CELL_COLS <= TMEM_COLS, "TMEM budget");
    static_assert(SPS == 1 || SPS == 2, "slabs per stage");
    static_assert(MW == 1 || MW == 2, "MMA warps");
};

// MXFP8 terms of h per regime (regime_nt_h() returns these): two everywhere, about 8 significant bits,
// the precision of a bf16 h. A third term (about 12 bits) was measured at 2-3 % more decode time and
// a third more W2 time in prefill.
constexpr int NTH_DECODE = 2, NTH_MID = 2, NTH_LARGE = 2;

// decode, <= 2 rows per expert on average
using W13Tiny = Cfg<0, 16, NT_X, 2, 5, 4, 6, 1, 2, 1024, NTH_DECODE>;
// W2 is bound by its activation ring as much as by its weight ring: five weight and five activation
// stages up to 512 experts (the shared memory for more experts' prefixes does not fit), four and
// four above
using W2Tiny = Cfg<1, 16, NTH_DECODE, 2, 5, 5, 6, 1, 2, 512>;
using W2TinyWideE = Cfg<1, 16, NTH_DECODE, 2, 4, 4, 6, 1, 2, 1024>;
// decode batches: <= 16 rows per expert
using W13Small = Cfg<0, 32, NT_X, 2, 4, 4, 6, 1, 2, 1024, NTH_DECODE>;
using W2Small = Cfg<1, 32, NTH_DECODE, 2, 4, 3, 4, 1, 2, 1024>;
// <= 64 rows per expert when H is not a multiple of 256 (else the stacked token-major tiles of gemm_rows.cu)
using W13Mid = Cfg<0, 64, NT_X, 2, 3, 3, 6, 1, 1, 1024, NTH_MID>;
using W2Mid = Cfg<1, 64, NTH_MID, 2, 3, 3, 6, 1, 1, 1024>;
// prefill
// (prefill weights are mostly re-read from L2, the activation rows are the bound: a third activation
// stage up to 512 experts, two above; with h in two terms W2 takes 96 token rows per tile like W13)
using W13Large = Cfg<0, 96, NT_X, 2, 2, 3, 4, 1, 1, 512, NTH_LARGE>;
using W2Large = Cfg<1, 96, NTH_LARGE, 2, 2, 3, 4, 1, 1, 512>;
using W13LargeWideE = Cfg<0, 96, NT_X, 2, 3, 2, 4, 1, 1, 1024, NTH_LARGE>;
using W2LargeWideE = Cfg<1, 96, NTH_LARGE, 2, 3, 2, 4, 1, 1>;
static_assert(W13Large::NMAX == 96 && W2Large::NMAX == 96 && W13Mid::NMAX == 64 && W2Mid::NMAX == 64,
              "regime_nmax() mirrors these");
static_assert(W13Tiny::NTO == W2Tiny::NT && W13Small::NTO == W2Small::NT && W13Mid::NTO == W2Mid::NT &&
                  W13Large::NTO == W2Large::NT && W13LargeWideE::NTO == W2LargeWideE::NT,
              "W2 reads as many h terms as W13 writes");


template <class C>
struct Smem {
    static constexpr int ASTAGE = C::SPS * SLAB_SMEM_BYTES;    // expanded E2M1 slabs
    static constexpr int BSLAB = C::NP * 128;                 // [term][row][128 K bytes]
    static constexpr int BSTAGE = C::SPS * BSLAB;
    static constexpr int BSSLAB = C::NP * 4;                  // B scale words [term][row] of one slab
    // a stage box writes its slabs' words back to back; a stage loaded slab by slab (across two
    // tiles) puts slab 1 at the next 128-byte boundary (tensor-copy destinations are 128-byte aligned)
    static constexpr int BSSLAB_PAD = (BSSLAB + 127) / 128 * 128;
    static constexpr int BSSTAGE = ((C::SPS - 1) * BSSLAB_PAD + BSSLAB + 127) / 128 * 128;
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
    // tile prefix [E + 1], scan scratch [32], then per expert its first padded row and its row count [E] each
    static constexpr size_t bytes(int E) { return 1024 + PREFIX_OFF + sizeof(int) * (size_t)(3 * E + 1 + 32); }
    static_assert(BSLAB % 1024 == 0 && ASTAGE % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
    static_assert(bytes(C::EMAX) <= 232448, "shared memory per CTA");
};




// FAST (W2 of the decode tiles only): the epilogue adds w * o into y with reduction atomics instead of
// writing the per-pair rows (MOE_FLAG_FAST_COMBINE); a separate instantiation, so the default kernels
// carry no code of it.
template <class C, bool FAST = false>
__global__ void __launch_bounds__(C::THREADS, 1) moe_gemm_kernel(const __grid_constant__ GemmParams p)
{
    constexpr int MODE = C::MODE, NMAX = C::NMAX, NT = C::NT, SPS = C::SPS, NP = C::NP;
    using S = Smem<C>;
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
    int *tile_start = reinterpret_cast<int *>(smem + S::PREFIX_OFF);
    int *scan_tmp = tile_start + p.E + 1;
    int *s_pad0 = scan_tmp + 32, *s_cnt = s_pad0 + p.E;   // per expert: first padded row, rows

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int E = p.E, MB = p.MB;

    // ---- tile prefix over experts (E <= 1024: four experts per thread)
    {
        int v[4];
        int s = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int e = tid * 4 + q;
            const int cnt = e < E ? (__ldg(p.offsets + e + 1) - __ldg(p.offsets + e)) : 0;
            if (e < E) {
                s_cnt[e] = cnt;
                s_pad0[e] = __ldg(p.padded + e);
            }
            v[q] = (cnt + NMAX - 1) / NMAX * MB;
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
        for (int q = 0; q < 4; ++q) {
            const int e = tid * 4 + q;
            if (e < E) tile_start[e] = run;
            run += v[q];
        }
        if (tid == C::THREADS - 1) tile_start[E] = run;   // the total
        __syncthreads();
    }
    const int total = tile_start[E];
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
    const int slabs = p.K / KSLAB;
    // This CTA's slabs, in order: tiles blockIdx.x, blockIdx.x + gridDim.x, ..., each with `slabs`
    // K-slabs; slab i sits in ring stage i / SPS at position i % SPS.
    const int my_tiles = (total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1;
    const int n_slabs = my_tiles * slabs;
    const uint64_t LIM = WAIT_LIMIT_NS;

    auto fail = [&]() {
        *s_abort = 1;
        record_error(p.dev_error, DEV_ERR_TIMEOUT);
    };
    // stage q (counted over this CTA's stages) has been consumed by its MMAs; nothing to wait for if q < 0
    auto wait_done = [&](int q) -> bool {
        return q < 0 || ptx::mbar_wait(&done[q % C::ND], (uint32_t)((q / C::ND) & 1), s_abort, LIM);
    };
    // first 128-element row of (tile, slab) in the 2-D view of the nibble region
    auto a_row = [&](const Tile &tl, int ka) { return ((tl.e * MB + tl.mb) * slabs + ka) * TILE_ROWS; };

    if (warp == 10) {
        // ===================== weight producer: per stage one TMA box of SPS slabs (E2M1 rows,
        // expanded in shared memory) and one bulk copy of their scales; two of each when the stage
        // straddles two tiles
        if (ptx::elect_one()) {
            ptx::prefetch_tmap(&p.tm_a);
            ptx::prefetch_tmap(&p.tm_a1);
        }
        __syncwarp();
        int ai = 0;
        uint32_t aph = 0;
        long long issued = 0;
        bool ok = true;
        int tcur = blockIdx.x, ka = 0;
        Tile tl = decode_tile<C::NMAX>(tcur, tile_start, E, MB, s_cnt, s_pad0);
        for (int i0 = 0; i0 < n_slabs; i0 += SPS) {
            if (!__all_sync(0xFFFFFFFFu, wait_done(i0 / SPS - C::NA))) { ok = false; break; }
            const int nsl = n_slabs - i0 < SPS ? n_slabs - i0 : SPS;
            if (ptx::elect_one()) {
                uint8_t *dst = aring + ai * S::ASTAGE;
                uint8_t *sdst = sfring + ai * S::SFSTAGE;
                // the TMA counts the bytes it reads (8 KB per slab), not the expanded 16 KB it writes
                ptx::mbar_arrive_expect_tx(&a_full[ai], (uint32_t)(nsl * (SLAB_NIB_BYTES + SLAB_SF_BYTES)));
                const int r0 = a_row(tl, ka);
                if (nsl == SPS && ka + SPS <= slabs) {
                    ptx::tma_load_2d(dst, &p.tm_a, 0, r0, &a_full[ai]);
                    ptx::bulk_g2s(sdst, p.wsf + (size_t)(r0 / TILE_ROWS) * SLAB_SF_BYTES,
                                  (uint32_t)(SPS * SLAB_SF_BYTES), &a_full[ai]);
                } else {
                    ptx::tma_load_2d(dst, &p.tm_a1, 0, r0, &a_full[ai]);
                    ptx::bulk_g2s(sdst, p.wsf + (size_t)(r0 / TILE_ROWS) * SLAB_SF_BYTES, SLAB_SF_BYTES, &a_full[ai]);
                    if (nsl == 2) {                  // the second slab opens the next tile
                        const Tile t2 = decode_tile<C::NMAX>(tcur + (int)gridDim.x, tile_start, E, MB, s_cnt, s_pad0);
                        const int r1 = a_row(t2, 0);
                        ptx::tma_load_2d(dst + SLAB_SMEM_BYTES, &p.tm_a1, 0, r1, &a_full[ai]);
                        ptx::bulk_g2s(sdst + SLAB_SF_BYTES, p.wsf + (size_t)(r1 / TILE_ROWS) * SLAB_SF_BYTES,
                                      SLAB_SF_BYTES, &a_full[ai]);
                    }
                }
            }
            __syncwarp();
            ++issued;
            ka += nsl;
            bool next_tile = false;
            while (ka >= slabs) {
                ka -= slabs;
                tcur += gridDim.x;
                next_tile = true;
            }
            if (next_tile && tcur < total) tl = decode_tile<C::NMAX>(tcur, tile_start, E, MB, s_cnt, s_pad0);
            if (++ai == C::NA) { ai = 0; aph ^= 1u; }
        }
        if (!ok && lane == 0) fail();
        volatile int never = 0;
        // drain: every issued copy must land before shared memory is released
        for (long long i = 1; i <= (issued < C::NA ? issued : C::NA); ++i) {
            const long long n = issued - i;
            __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&a_full[n % C::NA], (uint32_t)((n / C::NA) & 1), &never, LIM));
        }
    } else if (warp == 9) {
        // ===================== activation producer: per stage one 4-D TMA box of the term rows (128 K x
        // NMAX rows x NT terms x SPS slabs) and one 3-D box of their scale words (NMAX x NT x SPS); slab
        // by slab for a tile's last slab or a stage that crosses into the next tile
        if (ptx::elect_one()) {
            ptx::prefetch_tmap(&p.tm_b);
            ptx::prefetch_tmap(&p.tm_bs);
            ptx::prefetch_tmap(&p.tm_b1);
            ptx::prefetch_tmap(&p.tm_bs1);
        }
        // The activation terms come from the kernel before (gather, or W13 for W2): under
        // programmatic dependent launch everything above, and the weight producer's stream, may
        // run while that kernel finishes; this warp waits for it before its first copy.
        griddep_wait();
        if (lane == 0) griddep_launch_dependents();
        __syncwarp();
        int bi = 0;
        uint32_t bph = 0;
        long long issued = 0;
        bool ok = true;
        int tcur = blockIdx.x, ka = 0;
        Tile tl = decode_tile<C::NMAX>(tcur, tile_start, E, MB, s_cnt, s_pad0);
        for (int i0 = 0; i0 < n_slabs; i0 += SPS) {
            if (!__all_sync(0xFFFFFFFFu, wait_done(i0 / SPS - C::NB))) { ok = false; break; }
            const int nsl = n_slabs - i0 < SPS ? n_slabs - i0 : SPS;
            if (ptx::elect_one()) ptx::mbar_arrive_expect_tx(&b_full[bi], (uint32_t)(nsl * (S::BSLAB + S::BSSLAB)));
            if (nsl == SPS && ka + SPS <= slabs) {      // the stage's slabs in one box each for terms and scales
                if (ptx::elect_one()) {
                    ptx::tma_load_4d(bring + bi * S::BSTAGE, &p.tm_b, 0, tl.row0, 0, ka, &b_full[bi]);
                    ptx::tma_load_3d(bsring + bi * S::BSSTAGE, &p.tm_bs, tl.row0, 0, ka, &b_full[bi]);
                }
                __syncwarp();
                ka += SPS;
                if (ka == slabs) {
                    ka = 0;
                    tcur += gridDim.x;
                    if (tcur < total) tl = decode_tile<C::NMAX>(tcur, tile_start, E, MB, s_cnt, s_pad0);
                }
            } else {                                    // last slab of a tile, or a stage across two tiles
                for (int pos = 0; pos < nsl; ++pos) {
                    if (ptx::elect_one()) {
                        ptx::tma_load_4d(bring + bi * S::BSTAGE + pos * S::BSLAB, &p.tm_b1, 0, tl.row0, 0, ka, &b_full[bi]);
                        ptx::tma_load_3d(bsring + bi * S::BSSTAGE + pos * S::BSSLAB_PAD, &p.tm_bs1, tl.row0, 0, ka,
                                         &b_full[bi]);
                    }
                    __syncwarp();
                    if (++ka == slabs) {
                        ka = 0;
                        tcur += gridDim.x;
                        if (tcur < total) tl = decode_tile<C::NMAX>(tcur, tile_start, E, MB, s_cnt, s_pad0);
                    }
                }
            }
            ++issued;
            if (++bi == C::NB) { bi = 0; bph ^= 1u; }
        }
        if (!ok && lane == 0) fail();
        volatile int never = 0;
        for (long long i2 = 1; i2 <= (issued < C::NB ? issued : C::NB); ++i2) {
            const long long n = issued - i2;
            __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&b_full[n % C::NB], (uint32_t)((n / C::NB) & 1), &never, LIM));
        }
    } else if (warp >= 4 && warp < 8) {
        // ===================== scale-factor copiers: per stage, A's cells (weight stage) and B's cells
        // (one 32-bit word per B row: its 4 K-block scales; activation stage) of each slab into the
        // next TMEM cell, in this warp's lane quarter; lane r of every quarter holds rows r, r + 32,
        // ... in consecutive columns.
        int ai = 0, bi = 0, sc = 0;
        uint32_t aph = 0, bph = 0;
        bool ok = true;
        const uint32_t quarter = (uint32_t)((warp & 3) * 32) << 16;
        for (int i0 = 0; i0 < n_slabs; i0 += SPS) {
            const int nsl = n_slabs - i0 < SPS ? n_slabs - i0 : SPS;
            if (!__all_sync(0xFFFFFFFFu, wait_done(i0 / SPS - C::NSF) &&
                                             ptx::mbar_wait(&a_full[ai], aph, s_abort, LIM) &&
                                             ptx::mbar_wait(&b_full[bi], bph, s_abort, LIM))) { ok = false; break; }
            ptx::tc_fence_after();
            // the activation producer's test: one box for the stage (slab words back to back) or one per slab
            const bool whole = nsl == SPS && (i0 % slabs) + SPS <= slabs;
            for (int pos = 0; pos < nsl; ++pos) {
                const uint4 aw = *reinterpret_cast<const uint4 *>(sfring + ai * S::SFSTAGE + pos * SLAB_SF_BYTES + lane * 16);
                const uint32_t *bs = reinterpret_cast<const uint32_t *>(bsring + bi * S::BSSTAGE +
                                                                        pos * (whole ? S::BSSLAB : S::BSSLAB_PAD));
                const uint32_t cell = tmem + quarter + (uint32_t)(C::SF_BASE + sc * C::CELL_COLS + pos * C::SF_COLS);
                // the slab's cell in stores of 8 columns: A's 4, then one per 32 B rows (B row j: term
                // j / NMAX of token row j % NMAX), zeros in the columns no MMA reads
                uint32_t wv[C::SF_COLS];
                wv[0] = aw.x;
                wv[1] = aw.y;
                wv[2] = aw.z;
                wv[3] = aw.w;
#pragma unroll
                for (int c = 0; c < C::SF_COLS - 4; ++c) {
                    const int j = lane + 32 * c;
                    wv[4 + c] = (c < C::SFB_COLS && j < NP) ? bs[j] : 0u;
                }
#pragma unroll
                for (int c0 = 0; c0 < C::SF_COLS; c0 += 8) {
                    uint32_t v8[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) v8[q] = c0 + q < C::SF_COLS ? wv[c0 + q] : 0u;
                    if (c0 + 8 <= C::SF_COLS) {
                        ptx::tmem_st_32x32b_x8(cell + (uint32_t)c0, v8);
                    } else {
                        ptx::tmem_st_32x32b_x4(cell + (uint32_t)c0, v8[0], v8[1], v8[2], v8[3]);
                    }
                }
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sf_full[sc]);
            if (++ai == C::NA) { ai = 0; aph ^= 1u; }
            if (++bi == C::NB) { bi = 0; bph ^= 1u; }
            if (++sc == C::NSF) sc = 0;
        }
        if (!ok && lane == 0) fail();
    } else if (warp == 8 || (C::MW == 2 && warp == 11)) {
        // ===================== MMA issuers: stage s belongs to warp s % MW (s counted from the tile's
        // start when stages align with tiles, else over the CTA's whole stage sequence). The warp waits for the stage's
        // scale-factor cell only: the copiers fill it after the stage's weights and activations have
        // landed, so that one wait covers all three. One elected lane issues the stage's block-scaled MMAs
        // (four of K = 32 per slab) into the warp's own accumulator set and commits the stage to
        // done[s % ND]. Both warps walk every stage to follow the tiles: at a tile's start a warp waits
        // for the tile's accumulator buffer to be free, at its end it commits the tile (with or without
        // MMAs of its own in it), so the epilogue sees one arrival per warp and tile.
        const int q = warp == 8 ? 0 : 1;
        const uint64_t adesc0 = ptx::smem_desc_sw128(ptx::smem_u32(aring));
        const uint64_t bdesc0 = ptx::smem_desc_sw128(ptx::smem_u32(bring));
        int ai = 0, bi = 0, sc = 0, di = 0, ka = 0, st = 0, mine_in_tile = 0;
        uint32_t sph = 0, dph = 0;
        bool ok = true;
        // the four MMAs of slab `pos` of the current stage; kk0: this warp's 32-K blocks in the tile so far
        auto issue_slab = [&](int pos, int kk0) {
            const uint64_t ad = adesc0 + (uint64_t)((uint32_t)(ai * S::ASTAGE + pos * SLAB_SMEM_BYTES) >> 4);
            const uint64_t bd = bdesc0 + (uint64_t)((uint32_t)(bi * S::BSTAGE + pos * S::BSLAB) >> 4);
            const uint32_t sfa = tmem + (uint32_t)(C::SF_BASE + sc * C::CELL_COLS + pos * C::SF_COLS);
            const uint32_t dt0 = tmem + (uint32_t)((q * 2 + di) * C::D_COLS);
#pragma unroll
            for (int kb = 0; kb < 4; ++kb) {
                const int kk = kk0 + kb;
                // overwrite on the first use of each accumulator in the tile
                ptx::mma_mx_ss(dt0 + (uint32_t)((kk % C::NACC) * NP), ad + (uint64_t)(kb * 2), bd + (uint64_t)(kb * 2),
                               ptx::idesc_mx_e2m1_e4m3(128, NP, (uint32_t)kb), sfa, sfa + 4, kk >= C::NACC ? 1u : 0u);
            }
        };
        auto tile_start = [&]() -> bool {     // the tile's accumulators must be free
            if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&d_empty[di], dph ^ 1u, s_abort, LIM))) return false;
            ptx::tc_fence_after();
            mine_in_tile = 0;
            return true;
        };
        auto next_tile = [&]() {
            ka = 0;
            if (++di == 2) { di = 0; dph ^= 1u; }
        };
        for (int i0 = 0; i0 < n_slabs && ok; i0 += SPS, ++st) {
            const int nsl = n_slabs - i0 < SPS ? n_slabs - i0 : SPS;
            // when stages align with tiles, ownership counts stages from the tile's start, so the K split
            // between the two accumulator sets (and the rounding of their sum) does not depend on which
            // CTA ran the tile or on how many tiles it ran before
            const bool mine = (((slabs % SPS) == 0 ? ka / SPS : st) % C::MW) == q;
            if (mine) {
                if (!__all_sync(0xFFFFFFFFu, ptx::mbar_wait(&sf_full[sc], sph, s_abort, LIM))) { ok = false; break; }
                ptx::tc_fence_after();
            }
            if (ka + nsl <= slabs) {
                // the stage lies in one tile: one elected block for its MMAs and commits
                if (ka == 0 && !tile_start()) { ok = false; break; }
                const bool tile_end = ka + nsl == slabs;
                if (mine || tile_end) {
                    if (ptx::elect_one()) {
                        if (mine) {
#pragma unroll
                            for (int pos = 0; pos < SPS; ++pos)
                                if (pos < nsl) issue_slab(pos, mine_in_tile + 4 * pos);
                            ptx::mma_commit(&done[st % C::ND]);
                        }
                        if (tile_end) ptx::mma_commit(&d_full[di]);
                    }
                    __syncwarp();
                }
                if (mine) mine_in_tile += 4 * nsl;
                ka += nsl;
                if (ka == slabs) next_tile();
            } else {
                // the stage crosses into the next tile: slab by slab
                for (int pos = 0; pos < nsl; ++pos) {
                    if (ka == 0 && !tile_start()) { ok = false; break; }
                    const bool tile_end = ka == slabs - 1;
                    if (mine || tile_end) {
                        if (ptx::elect_one()) {
                            if (mine) issue_slab(pos, mine_in_tile);
                            if (tile_end) ptx::mma_commit(&d_full[di]);
                        }
                        __syncwarp();
                    }
                    if (mine) mine_in_tile += 4;
                    if (++ka == slabs) next_tile();
                }
                if (!ok) break;
                if (mine) {
                    if (ptx::elect_one()) ptx::mma_commit(&done[st % C::ND]);
                    __syncwarp();
                }
            }
            if (++ai == C::NA) ai = 0;
            if (++bi == C::NB) bi = 0;
            if (++sc == C::NSF) { sc = 0; sph ^= 1u; }
        }
        if (!ok && lane == 0) fail();
        // one arrival per MMA warp once its MMAs have retired (TMEM is released after that)
        volatile int never = 0;
        if (ptx::elect_one()) ptx::mma_commit(mma_done);
        __syncwarp();
        if (q == 0) __all_sync(0xFFFFFFFFu, ptx::mbar_wait(mma_done, 0, &never, LIM));
    } else if (warp < 4) {
        // ===================== epilogue: TMEM -> registers -> global. The W13 epilogue pairs warps
        // at a named barrier, so no warp leaves the tile loop early: after a failed wait a warp
        // skips the work but still meets its partner at every barrier.
        const uint32_t t_lane = (uint32_t)(warp * 32) << 16;
        int di = 0, chunk = 0;
        uint32_t dph = 0;
        bool ok = true;
        int j = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x, ++j) {
            const Tile tl = decode_tile<C::NMAX>(t, tile_start, E, MB, s_cnt, s_pad0);
            // MMA warp q wrote into the tile iff one of the tile's stages is one of its stages
            const int s_first = (j * slabs) / SPS, s_last = (j * slabs + slabs - 1) / SPS;
            const unsigned wrote = (C::MW == 1 || s_last > s_first) ? ((1u << C::MW) - 1u)
                                 : (slabs % SPS) == 0        ? 1u
                                                             : (1u << (s_first % C::MW));
            ok = ok && __all_sync(0xFFFFFFFFu, ptx::mbar_wait(&d_full[di], dph, s_abort, LIM));
            ptx::tc_fence_after();
            for (int c0 = 0; c0 < tl.n; c0 += 16, ++chunk) {
                uint32_t raw[16];
#pragma unroll
                for (int q = 0; q < 16; ++q) raw[q] = 0u;
                if (ok) {
                    // sum the term columns of every accumulator of every MMA warp that wrote the tile, in
                    // (warp, accumulator, term) order; loads go out in groups of four with one wait each
                    constexpr int NCOMB = C::MW * C::NACC * NT, G = 4;
#pragma unroll
                    for (int g0 = 0; g0 < NCOMB; g0 += G) {
                        uint32_t part[G][16];
#pragma unroll
                        for (int u = 0; u < G; ++u) {
                            const int idx = g0 + u, w = idx / (C::NACC * NT), a = (idx / NT) % C::NACC, term = idx % NT;
                            if (idx < NCOMB && ((wrote >> w) & 1u))
                                ptx::tmem_ld_32x32b_x16(tmem + t_lane + (uint32_t)((w * 2 + di) * C::D_COLS + a * NP +
                                                                                    term * NMAX + c0), part[u]);
                        }
                        ptx::tmem_wait_ld();
#pragma unroll
                        for (int u = 0; u < G; ++u) {
                            const int idx = g0 + u, w = idx / (C::NACC * NT);
                            if (idx < NCOMB && ((wrote >> w) & 1u))
#pragma unroll
                                for (int q = 0; q < 16; ++q)
                                    raw[q] = __float_as_uint(__uint_as_float(raw[q]) + __uint_as_float(part[u][q]));
                        }
                    }
                }
                if (MODE == 0) {
                    // lane i < 16: gate of feature f; lane i + 16: up of the same f. Lane i ends with
                    // h[f] for tokens c0 .. c0+7, lane i + 16 for tokens c0+8 .. c0+15.
                    const bool is_gate = lane < 16;
                    const int f = tl.mb * 64 + warp * 16 + (lane & 15);
                    const float L = p.swiglu_limit;
                    float h[8], am[8];
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
                        h[j] = silu_f(gt) * up;
                        am[j] = fabsf(h[j]);
                    }
                    // W2 scale blocks are 32 consecutive features: 16 in this half-warp, 16 in the
                    // partner warp (warps 0+1 and 2+3), which trade maxima through shared memory
#pragma unroll
                    for (int j = 0; j < 8; ++j)
#pragma unroll
                        for (int o = 1; o < 16; o <<= 1) am[j] = fmaxf(am[j], __shfl_xor_sync(0xFFFFFFFFu, am[j], o));
                    float *pm = pairmax + (chunk & 1) * 64;
                    if ((lane & 15) == 0)
#pragma unroll
                        for (int j = 0; j < 8; ++j) pm[warp * 16 + (lane >> 4) * 8 + j] = am[j];
                    ptx::bar_sync_n(1 + (warp >> 1), 64);
                    if (ok) {
                        const int blk = f >> 5;                      // W2 K-block of this feature
                        const bool writes_scale = (lane & 15) == 0 && (warp & 1) == 0;
#pragma unroll
                        for (int j = 0; j < 8; j += 2) {           // two token rows per conversion
                            const float *pmj = pm + (warp ^ 1) * 16 + (lane >> 4) * 8 + j;
                            const int e0 = mxfp8_block_exp(fmaxf(am[j], pmj[0]));
                            const int e1 = mxfp8_block_exp(fmaxf(am[j + 1], pmj[1]));
                            const int64_t row = (int64_t)tl.row0 + c0 + (lane >> 4) * 8 + j;
                            float r0 = h[j], r1 = h[j + 1];
#pragma unroll
                            for (int term = 0; term < C::NTO; ++term) {
                                uint32_t sb0, sb1;
                                const uint32_t q = mxfp8_term_2x(r0, r1, e0, e1, term, sb0, sb1);
                                uint8_t *dq = p.hq + (((int64_t)(f >> 7) * C::NTO + term) * p.rows_cap + row) * 128 + (f & 127);
                                dq[0] = (uint8_t)q;
                                dq[128] = (uint8_t)(q >> 8);
                                if (writes_scale) {
                                    uint8_t *ds = p.hs + (((int64_t)(blk >> 2) * C::NTO + term) * p.rows_sf + row) * 4 + (blk & 3);
                                    ds[0] = (uint8_t)sb0;
                                    ds[4] = (uint8_t)sb1;
                                }
                            }
                        }
                    }
                } else if (ok) {
                    const int c = tl.mb * TILE_ROWS + warp * 32 + lane;
                    const int my_pair = (lane < 16) ? __ldg(p.row_to_pair + tl.row0 + c0 + lane) : -1;
                    if constexpr (FAST) {
                        // fast combine: w * o added into the token's row of y; lane j < 16 holds row j's weight
                        const float my_w = (my_pair >= 0 && my_pair < p.P) ? __ldg(p.topk_w + my_pair) : 0.f;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int pr = __shfl_sync(0xFFFFFFFFu, my_pair, j);
                            const float wj = __shfl_sync(0xFFFFFFFFu, my_w, j);
                            if (pr >= 0 && pr < p.P)
                                ptx::red_add_f32(p.y + (int64_t)(pr / p.k) * p.H + c, wj * __uint_as_float(raw[j]));
                            else if (pr >= p.P && lane == 0)
                                record_error(p.dev_error, DEV_ERR_ID_RANGE);
                        }
                    } else {
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

// The fast combine adds into y: the gather kernel that runs first zeroes it (n4 float4 words; y is
// 16-byte aligned), which the W2 GEMM, two launches later, sees complete.
__device__ __forceinline__ void zero_y(float *y, int64_t n4)
{
    if (!y) return;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x)
        reinterpret_cast<float4 *>(y)[i] = z;
}

// Gathered activations as NT_X MXFP8 terms: row r of the permutation gets
// the terms of x[token(r)]. Padding rows (row_to_pair == -1) are not written:
// every GEMM row is computed from its own activation row only (MMA rows, the
// 32-feature block maxima of h, the epilogue stores), and outputs of padding
// rows are never stored, so their contents do not matter. One
// thread per (row, 32-element block). Terms are E4M3 bytes
// [H/128][NT_X][rows_cap][128] (slab-major: one TMA box fetches the slabs of a
// stage for all rows and terms of a tile); scales are 32-bit words
// [H/128][NT_X][rows_sf], byte b % 4 of word (b / 4, t, r) for 32-element
// block b. Rows past padded[E] are not touched.
// A thread stores its block's 32 term bytes with one 32-byte store per term
// (whole sectors); the four threads of a scale word (consecutive blocks of one
// row: H / 32 is a multiple of 4) hand their bytes to the first, which stores
// the word. Every warp runs the same number of iterations (lanes past the end
// only skip the stores), so the shuffles always see the whole warp.
__global__ void gather_quant_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ row_to_pair,
                                    const int32_t *__restrict__ padded, int E, int H, int k, int64_t P,
                                    int64_t rows_cap, int64_t rows_sf, uint8_t *__restrict__ xq,
                                    uint8_t *__restrict__ xs, int32_t *dev_error, float *y_zero, int64_t y_n4,
                                    uint32_t *zero_counts)
{
    griddep_wait();                  // the permutation (and x) come from earlier kernels
    // The forward's device error word and the fused decode GEMMs' per-expert counters are reset only
    // now: a kernel of the previous call may run until this wait returns (the fused decode kernel
    // lets its successor start early). Every kernel of this call that records an error or counts
    // tiles waits for this grid to complete first.
    if (blockIdx.x == 0 && threadIdx.x == 0) *dev_error = 0;
    if (zero_counts && blockIdx.x == 0)
        for (int e = threadIdx.x; e < E; e += blockDim.x) zero_counts[e] = 0u;
    griddep_launch_dependents();
    zero_y(y_zero, y_n4);
    const int64_t R = __ldg(padded + E);
    const int nblk = H / 32;
    const int64_t n = R * nblk;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) & ~(int64_t)31;
    const int lane = threadIdx.x & 31;
    for (int64_t wbase = warp0; wbase < n; wbase += stride) {
        const int64_t idx = wbase + lane;
        const bool live = idx < n;
        const int64_t r = live ? idx / nblk : 0;
        const int b = live ? (int)(idx - r * nblk) : 0;
        const int32_t pr = live ? __ldg(row_to_pair + r) : -1;
        const bool real = live && pr >= 0 && pr < P;
        float v[32];
        if (real) {
            const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)(pr / k) * H + b * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 u = __ldg(src + q);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    v[q * 8 + 2 * z] = __uint_as_float(w[z] << 16);
                    v[q * 8 + 2 * z + 1] = __uint_as_float(w[z] & 0xFFFF0000u);
                }
            }
        }
        float mx = 0.f;
        if (real) {
#pragma unroll
            for (int q = 0; q < 32; ++q) mx = fmaxf(mx, fabsf(v[q]));
        }
        const int e1 = mxfp8_block_exp(mx);
#pragma unroll
        for (int t = 0; t < NT_X; ++t) {
            uint32_t wq[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u}, sbyte = 0;
            if (real) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const uint32_t lo = mxfp8_term_pair(v[4 * q], v[4 * q + 1], e1, t, sbyte);
                    const uint32_t hi = mxfp8_term_pair(v[4 * q + 2], v[4 * q + 3], e1, t, sbyte);
                    wq[q] = lo | (hi << 16);
                }
            }
            // the scale word of blocks 4j .. 4j+3: lane (b % 4 == 0) collects its three neighbours' bytes
            uint32_t word = sbyte;
            word |= __shfl_down_sync(0xFFFFFFFFu, sbyte, 1) << 8;
            word |= __shfl_down_sync(0xFFFFFFFFu, sbyte, 2) << 16;
            word |= __shfl_down_sync(0xFFFFFFFFu, sbyte, 3) << 24;
            if (real) {
                ptx::st_global_v8(xq + (((int64_t)(b >> 2) * NT_X + t) * rows_cap + r) * 128 + (b & 3) * 32, wq);
                if ((b & 3) == 0)
                    *reinterpret_cast<uint32_t *>(xs + (((int64_t)(b >> 2) * NT_X + t) * rows_sf + r) * 4) = word;
            }
        }
    }
}

// Gather in two passes for batches with many rows per expert, where the one-pass gather above would
// convert every token's x k times (once per row). Pass 1, one warp per row: a real row records itself
// in the inverse map p2r[pair] = row (padding rows are left as they are, see above). Pass 2, one
// thread per (token, 32-element block) as above: the block's terms are computed once and stored to
// each of the token's k rows. p2r lives in the fp32 staging region, which only the W2 GEMM writes
// later; an entry is trusted only if row_to_pair sends its row back to the pair (a pair without a row,
// i.e. with an expert id the permutation skipped, keeps whatever the region held).
__global__ void gather_rows_kernel(const int32_t *__restrict__ row_to_pair, const int32_t *__restrict__ padded,
                                   int E, int64_t P, int32_t *__restrict__ p2r, int32_t *dev_error, float *y_zero,
                                   int64_t y_n4)
{
    griddep_wait();                  // the permutation comes from an earlier kernel
    if (blockIdx.x == 0 && threadIdx.x == 0) *dev_error = 0;   // the forward's error word, as above
    griddep_launch_dependents();
    zero_y(y_zero, y_n4);
    const int64_t R = __ldg(padded + E);
    for (int64_t r = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; r < R; r += (int64_t)gridDim.x * blockDim.x) {
        const int32_t pr = __ldg(row_to_pair + r);
        if (pr >= 0 && pr < P) p2r[pr] = (int32_t)r;   // entries >= P are recorded by the W2 GEMM
    }
}

__global__ void gather_tokens_kernel(const uint16_t *__restrict__ x, const int32_t *__restrict__ row_to_pair,
                                     const int32_t *__restrict__ padded, const int32_t *__restrict__ p2r, int E,
                                     int T, int H, int k, int64_t rows_cap, int64_t rows_sf,
                                     uint8_t *__restrict__ xq, uint8_t *__restrict__ xs)
{
    griddep_wait();                  // the inverse map and the padding rows come from the kernel before
    griddep_launch_dependents();
    const int64_t R = __ldg(padded + E);
    const int nblk = H / 32;
    const int64_t n = (int64_t)T * nblk;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t warp0 = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) & ~(int64_t)31;
    const int lane = threadIdx.x & 31;
    for (int64_t wbase = warp0; wbase < n; wbase += stride) {
        const int64_t idx = wbase + lane;
        const bool live = idx < n;
        const int64_t t = live ? idx / nblk : 0;
        const int b = live ? (int)(idx - t * nblk) : 0;
        float v[32];
        float mx = 0.f;
        if (live) {
            const uint4 *src = reinterpret_cast<const uint4 *>(x + t * H + b * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint4 u = __ldg(src + q);
                const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                for (int z = 0; z < 4; ++z) {
                    v[q * 8 + 2 * z] = __uint_as_float(w[z] << 16);
                    v[q * 8 + 2 * z + 1] = __uint_as_float(w[z] & 0xFFFF0000u);
                }
            }
#pragma unroll
            for (int q = 0; q < 32; ++q) mx = fmaxf(mx, fabsf(v[q]));
        }
        const int e1 = mxfp8_block_exp(mx);
        uint32_t wq[NT_X][8], word[NT_X];
#pragma unroll
        for (int tt = 0; tt < NT_X; ++tt) {
            uint32_t sbyte = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                if (live) {
                    const uint32_t lo = mxfp8_term_pair(v[4 * q], v[4 * q + 1], e1, tt, sbyte);
                    const uint32_t hi = mxfp8_term_pair(v[4 * q + 2], v[4 * q + 3], e1, tt, sbyte);
                    wq[tt][q] = lo | (hi << 16);
                } else {
                    wq[tt][q] = 0u;
                }
            }
            word[tt] = sbyte;
            word[tt] |= __shfl_down_sync(0xFFFFFFFFu, sbyte, 1) << 8;
            word[tt] |= __shfl_down_sync(0xFFFFFFFFu, sbyte, 2) << 16;
            word[tt] |= __shfl_down_sync(0xFFFFFFFFu, sbyte, 3) << 24;
        }
        if (!live) continue;
        for (int j = 0; j < k; ++j) {
            const int64_t p = t * k + j;
            const int32_t r = __ldg(p2r + p);
            if (!(r >= 0 && r < R) || __ldg(row_to_pair + r) != (int32_t)p) continue;   // no row for this pair
#pragma unroll
            for (int tt = 0; tt < NT_X; ++tt) {
                ptx::st_global_v8(xq + (((int64_t)(b >> 2) * NT_X + tt) * rows_cap + r) * 128 + (b & 3) * 32, wq[tt]);
                if ((b & 3) == 0)
                    *reinterpret_cast<uint32_t *>(xs + (((int64_t)(b >> 2) * NT_X + tt) * rows_sf + r) * 4) = word[tt];
            }
        }
    }
}

// y[t, c] = sum_j w[t, j] * staging[t*k + j, c], slots in ascending order, in fp32; BF16: y is stored as
// bf16 bits, the fp32 sum rounded to nearest even.
template <bool BF16>
__global__ void combine_kernel(const float *__restrict__ staging, const float *__restrict__ w, int T, int H,
                               int k, void *__restrict__ y)
{
    griddep_wait();                  // staging comes from the W2 GEMM
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
        if (BF16) {
            const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 v;
            v.x = *reinterpret_cast<const uint32_t *>(&lo);
            v.y = *reinterpret_cast<const uint32_t *>(&hi);
            reinterpret_cast<uint2 *>(static_cast<uint16_t *>(y) + t * H)[c4] = v;
        } else {
            reinterpret_cast<float4 *>(static_cast<float *>(y) + t * H)[c4] = acc;
        }
    }
}

template <class C, bool FAST = false>
cudaError_t launch_gemm(const GemmParams &p, int grid, cudaStream_t s, bool pdl)
{
    static unsigned long long attr_set = 0;   // bit d: attribute set on device d
    const size_t smem = Smem<C>::bytes(p.E);
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 64 || !((attr_set >> dev) & 1ull)) {
        cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<C, FAST>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)Smem<C>::bytes(C::EMAX));
        if (e != cudaSuccess) return e;
        if (dev < 64) __atomic_fetch_or(&attr_set, 1ull << dev, __ATOMIC_RELAXED);
    }
    return launch_ex(moe_gemm_kernel<C, FAST>, dim3(grid), dim3(C::THREADS), smem, s, pdl, p);
}

}  // namespace

Regime pick_regime(int T, int k, int E, int H)
{
    const double avg = (double)T * k / E;
    if (avg <= 2.0) return Regime::Tiny;
    if (avg <= 16.0) return Regime::Small;
    if (avg <= 64.0) return Regime::Mid;      // stacked 64-row token-major tiles, or weight-major 64-row ones
    if (H % 256 != 0) return Regime::Large;   // weight-major 96-row tiles
    return Regime::Huge;       // token-major tiles (gemm_rows.cu): 256 W2 output rows per tile
}

int regime_nmax(Regime rg, int which)
{
    (void)which;
    switch (rg) {
    case Regime::Tiny: return 16;
    case Regime::Small: return 32;
    case Regime::Mid: return 64;
    case Regime::Large: return 96;
    default: return 128;
    }
}

int regime_nt_h(Regime rg)
{
    switch (rg) {
    case Regime::Tiny:
    case Regime::Small: return NTH_DECODE;
    case Regime::Mid: return NTH_MID;
    default: return NTH_LARGE;
    }
}

int regime_sps(Regime rg) { return rg == Regime::Huge ? 1 : 2; }

static void mark(const ForwardArgs &a, int i, cudaStream_t s)
{
    if (a.events && a.events[i]) cudaEventRecord(static_cast<cudaEvent_t>(a.events[i]), s);
}

ForwardPlan plan_forward(Regime rg, int H, int I, int E, bool fast_flag, bool y_bf16, bool split_gemms)
{
    ForwardPlan pl;
    pl.two_pass = rg == Regime::Mid || rg == Regime::Large || rg == Regime::Huge;
    // The flag permits the atomic combine; it is taken where it measured faster, up to 16 rows per
    // expert on average (the weight-major decode tiles). Larger batches keep the slot-ordered combine:
    // their W2 epilogues would issue T*k*H reductions, which cost the L2 more than the per-pair rows'
    // round trip.
    pl.fast = fast_flag && !y_bf16 && (rg == Regime::Tiny || rg == Regime::Small);
    // The smallest batches run both GEMMs in one persistent launch (gemm_decode.cu), unless an event
    // is to be recorded between them.
    pl.fused = rg == Regime::Tiny && !split_gemms && decode_fused_supported(H, I, E);
    pl.launches = (pl.two_pass ? 2 : 1) + (pl.fused ? 1 : 2) + (pl.fast ? 0 : 1);
    return pl;
}

cudaError_t launch_forward(const ForwardArgs &a, cudaStream_t s)
{
    const int64_t P = (int64_t)a.T * a.k;
    cudaError_t err;
    // Kernels after the first overlap their start with the end of the one before (programmatic
    // dependent launch), except when events are recorded between them to time each kernel alone.
    bool pdl = true;
    for (int i = 0; i < 5 && a.events; ++i)
        if (a.events[i]) pdl = false;
    const ForwardPlan pl = plan_forward(a.regime, a.H, a.I, a.E, a.fast_combine, a.y_bf16,
                                        a.events && a.events[2]);
    mark(a, 0, s);
    const bool fast = pl.fast, two_pass = pl.two_pass, fused = pl.fused;
    float *y_zero = fast ? static_cast<float *>(a.y) : nullptr;
    const int64_t y_n4 = (int64_t)a.T * a.H / 4;
    if (two_pass) {
        int32_t *p2r = reinterpret_cast<int32_t *>(a.staging);     // P entries; W2 overwrites them later
        int grid = (int)((a.rows_cap + 255) / 256);                  // a thread per row
        if (grid > 8 * 1024) grid = 8 * 1024;
        err = launch_ex(gather_rows_kernel, dim3(grid), dim3(256), 0, s, pdl, a.row_to_pair, a.padded, a.E, P, p2r,
                        a.dev_error, y_zero, y_n4);
        if (err != cudaSuccess) return err;
        const int64_t n = (int64_t)a.T * (a.H / 32);
        grid = (int)((n + 255) / 256);
        if (grid > 8 * 1024) grid = 8 * 1024;
        if (grid < 1) grid = 1;
        err = launch_ex(gather_tokens_kernel, dim3(grid), dim3(256), 0, s, pdl, a.x, a.row_to_pair, a.padded,
                        (const int32_t *)p2r, a.E, a.T, a.H, a.k, a.rows_cap, a.rows_sf, a.xq, a.xs);
        if (err != cudaSuccess) return err;
    } else {
        const int64_t n = a.rows_cap * (a.H / 32);
        int grid = (int)((n + 255) / 256);
        if (grid > 8 * 1024) grid = 8 * 1024;
        if (grid < 1) grid = 1;
        err = launch_ex(gather_quant_kernel, dim3(grid), dim3(256), 0, s, pdl, a.x, a.row_to_pair, a.padded, a.E,
                        a.H, a.k, P, a.rows_cap, a.rows_sf, a.xq, a.xs, a.dev_error, y_zero, y_n4,
                        fused ? a.done13 : nullptr);
        if (err != cudaSuccess) return err;
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
    g.rows_cap = a.rows_cap;
    g.rows_sf = a.rows_sf;
    g.hq = a.hq;
    g.hs = a.hs;
    g.staging = a.staging;
    g.y = nullptr;                    // W13 writes h; only W2 may add into y
    g.topk_w = a.topk_w;
    g.dev_error = a.dev_error;

    // W13: K = H, 64 features (128 rows) per weight tile
    g.tm_a = a.tmap_w13;
    g.tm_a1 = a.tmap_w13_1;
    g.tm_b = a.tmap_xq;
    g.tm_b1 = a.tmap_xq1;
    g.tm_bs = a.tmap_xs;
    g.tm_bs1 = a.tmap_xs1;
    g.wsf = a.packed + (size_t)a.E * 2 * a.I * (a.H / 2);
    g.K = a.H;
    g.MB = a.I / 64;
    const Regime rg = a.regime;
    // 17 to 64 rows per expert: token-major tiles of 64 token rows x 2 stacked terms where the 256-row
    // weight blocks divide H (gemm_rows.cu), else the 64-row weight-major tiles
    const bool rows64 = rg == Regime::Mid && a.H % 256 == 0;
    if (fused) {
        GemmParams g2 = g;
        g2.y = fast ? static_cast<float *>(a.y) : nullptr;
        g2.tm_a = a.tmap_w2;
        g2.tm_a1 = a.tmap_w2_1;
        g2.tm_b = a.tmap_hq;
        g2.tm_b1 = a.tmap_hq1;
        g2.tm_bs = a.tmap_hs;
        g2.tm_bs1 = a.tmap_hs1;
        g2.wsf = a.packed + packed_w13_bytes(a.E, a.H, a.I) + (size_t)a.E * a.H * (a.I / 2);
        g2.K = a.I;
        g2.MB = a.H / TILE_ROWS;
        if (a.rows8) {                 // at most 8 tokens: 8-row tiles (no expert holds more rows)
            g.tm_b = a.tmap_xq8;
            g.tm_bs = a.tmap_xs8;
            g2.tm_b = a.tmap_hq8;
            g2.tm_bs = a.tmap_hs8;
        }
        err = launch_gemm_decode(g, g2, a.done13, fast, a.rows8, a.num_sms, s, pdl);
        if (err != cudaSuccess) return err;
    }
    err = fused               ? cudaSuccess
        : rg == Regime::Huge  ? launch_gemm_rows(g, 0, false, a.num_sms, s, pdl)
        : rows64              ? launch_gemm_rows(g, 0, true, a.num_sms, s, pdl)
        : rg == Regime::Tiny  ? launch_gemm<W13Tiny>(g, a.num_sms, s, pdl)
        : rg == Regime::Small ? launch_gemm<W13Small>(g, a.num_sms, s, pdl)
        : rg == Regime::Mid   ? launch_gemm<W13Mid>(g, a.num_sms, s, pdl)
                              : (a.E <= W13Large::EMAX ? launch_gemm<W13Large>(g, a.num_sms, s, pdl)
                                                       : launch_gemm<W13LargeWideE>(g, a.num_sms, s, pdl));
    if (err != cudaSuccess) return err;
    mark(a, 2, s);

    // W2: K = I, 128 output features per weight tile
    g.y = fast ? static_cast<float *>(a.y) : nullptr;
    g.tm_a = a.tmap_w2;
    g.tm_a1 = a.tmap_w2_1;
    g.tm_b = a.tmap_hq;
    g.tm_b1 = a.tmap_hq1;
    g.tm_bs = a.tmap_hs;
    g.tm_bs1 = a.tmap_hs1;
    g.wsf = a.packed + packed_w13_bytes(a.E, a.H, a.I) + (size_t)a.E * a.H * (a.I / 2);
    g.K = a.I;
    g.MB = a.H / TILE_ROWS;
    err = fused               ? cudaSuccess
        : rg == Regime::Huge  ? launch_gemm_rows(g, 1, false, a.num_sms, s, pdl)
        : rows64              ? launch_gemm_rows(g, 1, true, a.num_sms, s, pdl)
        : rg == Regime::Tiny  ? (a.E <= W2Tiny::EMAX ? (fast ? launch_gemm<W2Tiny, true>(g, a.num_sms, s, pdl)
                                                          : launch_gemm<W2Tiny>(g, a.num_sms, s, pdl))
                                                     : (fast ? launch_gemm<W2TinyWideE, true>(g, a.num_sms, s, pdl)
                                                          : launch_gemm<W2TinyWideE>(g, a.num_sms, s, pdl)))
        : rg == Regime::Small ? (fast ? launch_gemm<W2Small, true>(g, a.num_sms, s, pdl)
                                      : launch_gemm<W2Small>(g, a.num_sms, s, pdl))
        : rg == Regime::Mid   ? launch_gemm<W2Mid>(g, a.num_sms, s, pdl)
                              : (a.E <= W2Large::EMAX ? launch_gemm<W2Large>(g, a.num_sms, s, pdl)
                                                      : launch_gemm<W2LargeWideE>(g, a.num_sms, s, pdl));
    if (err != cudaSuccess) return err;
    mark(a, 3, s);
    if (!fast) {                     // the fast combine has already added every pair into y
        const int64_t n = (int64_t)a.T * (a.H / 4);
        int grid = (int)((n + 255) / 256);
        if (grid > 4 * 1024) grid = 4 * 1024;
        if (grid < 1) grid = 1;
        err = a.y_bf16 ? launch_ex(combine_kernel<true>, dim3(grid), dim3(256), 0, s, pdl, (const float *)a.staging,
                                   a.topk_w, a.T, a.H, a.k, a.y)
                       : launch_ex(combine_kernel<false>, dim3(grid), dim3(256), 0, s, pdl, (const float *)a.staging,
                                   a.topk_w, a.T, a.H, a.k, a.y);
        if (err != cudaSuccess) return err;
    }
    mark(a, 4, s);
    note_launch(pl.launches);
    return cudaSuccess;
}

}  // namespace moe

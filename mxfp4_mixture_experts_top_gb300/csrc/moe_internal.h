// Internal declarations shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace moe {

// Device error codes (same values as moe_status_t in the public header).
constexpr int DEV_ERR_ID_RANGE = 6;   // MOE_ERR_DEVICE
constexpr int DEV_ERR_TIMEOUT = 7;    // MOE_ERR_TIMEOUT

// Activations enter the block-scaled GEMMs as sums of MXFP8 terms (mxfp8_terms.cuh):
// x (bf16) in NT_X terms, h (fp32 SiLU(gate)*up) in regime_nt_h() terms.
constexpr int NT_X = 2;

// GEMM tile shapes by the average rows per expert (T*k/E): decode batches get
// small tiles with deep pipelines, prefill batches large tiles.
enum class Regime { Tiny, Small, Mid, Large, Huge };
Regime pick_regime(int T, int k, int E, int H);
int regime_nmax(Regime rg, int which);   // token rows per tile; which 0: W13, 1: W2
int regime_sps(Regime rg);               // K-slabs per weight stage
// MXFP8 terms of h (gemm.cu sets them per tile regime; currently two, about 8 significant bits, the
// precision of a bf16 h).
int regime_nt_h(Regime rg);

// Programmatic dependent launch. A kernel launched with `pdl` may start while
// the previous kernel of the stream still runs. Before it reads or writes
// anything that kernel, or any earlier work, produces or reads, it executes
// griddep_wait(), which returns once the earlier grids have completed and
// their memory is visible. A kernel signals griddep_launch_dependents() only
// after its own griddep_wait(), so the part of a kernel that runs before its
// wait overlaps the one kernel before it, never an earlier one.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_ex(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                             Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

#ifdef __CUDACC__
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
#endif

// Bounded pipeline waits give up after this much wall time.
constexpr unsigned long long WAIT_LIMIT_NS = 2000000000ull;   // 2 s

void note_launch(int n);

cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                         uint32_t *bitmatrix, cudaStream_t s);

cudaError_t launch_permute(const int32_t *ids, int T, int E, int k, int block_m, int32_t *counts,
                           int32_t *offsets, int32_t *padded, int32_t *row_to_pair, int64_t rows_cap,
                           int32_t *pair_to_row, int32_t *dev_error, cudaStream_t s);

// Routing and permutation in one launch (one thread block) up to this many tokens; two launches above.
constexpr int ROUTE_PERMUTE_FUSED_MAX_T = 128;

cudaError_t launch_route_permute(const float *logits, int T, int E, int k, int block_m, int32_t *ids, float *w,
                                 uint32_t *bitmatrix, int32_t *counts, int32_t *offsets, int32_t *padded,
                                 int32_t *row_to_pair, int64_t rows_cap, int32_t *pair_to_row, int32_t *dev_error,
                                 cudaStream_t s);

cudaError_t launch_prepack(const uint8_t *w13_q, const uint8_t *w13_s, const uint8_t *w2_q,
                           const uint8_t *w2_s, int E, int H, int I, uint8_t *packed, cudaStream_t s);

cudaError_t launch_dequant(const uint8_t *packed, int which, int expert, int E, int H, int I,
                           uint16_t *out, cudaStream_t s);

// Offsets (bytes) of the two prepacked matrices inside the packed buffer.
size_t packed_w13_bytes(int E, int H, int I);
size_t packed_w2_bytes(int E, int H, int I);

struct ForwardArgs {
    int T, H, I, E, k, block_m;
    float swiglu_limit;
    bool fast_combine;           // MOE_FLAG_FAST_COMBINE given: the decode tiles' W2 adds w * o into y
    int64_t rows_cap, rows_sf;   // permutation rows; rows of the scale-word arrays (a multiple of 4)
    const uint16_t *x;
    const uint8_t *packed;
    const float *topk_w;
    const int32_t *offsets, *padded, *row_to_pair;
    void *y;                     // fp32 [T, H], or bf16 bits with y_bf16
    bool y_bf16;
    int32_t *dev_error;
    uint32_t *done13;      // [E] per-expert W13 tiles finished (the fused decode GEMMs), in the workspace
    uint8_t *xq, *xs;      // x terms [H/128][NT_X][rows_cap][128], scale words [H/128][NT_X][rows_sf]
    uint8_t *hq, *hs;      // h terms [I/128][nt_h][rows_cap][128], scale words [I/128][nt_h][rows_sf]
    float *staging;
    CUtensorMap tmap_w13, tmap_w13_1, tmap_w2, tmap_w2_1;   // weight nibbles: stage / single-slab boxes
    CUtensorMap tmap_xq, tmap_xq1, tmap_hq, tmap_hq1;      // activation terms: stage / one-slab boxes
    CUtensorMap tmap_xs, tmap_xs1, tmap_hs, tmap_hs1;      // their scale words
    bool rows8;            // T <= 8: the maps below (8-row boxes of a whole stage) are set
    CUtensorMap tmap_xq8, tmap_xs8, tmap_hq8, tmap_hs8;
    Regime regime;
    int num_sms;
    void *const *events;   // optional: 5 cudaEvent_t recorded between kernels
};

// What a forward launches for one layer shape (the single place that decides it).
struct ForwardPlan {
    bool two_pass;   // gather in two kernels (inverse map, then one conversion per token)
    bool fused;      // W13 and W2 in one persistent launch (gemm_decode.cu)
    bool fast;       // W2 adds w * o into y with reduction atomics; no combine kernel
    int launches;    // kernels launched
};
// split_gemms: an event is recorded between the W13 and the W2 GEMM, so they stay two launches.
ForwardPlan plan_forward(Regime rg, int H, int I, int E, bool fast_flag, bool y_bf16, bool split_gemms);

cudaError_t launch_forward(const ForwardArgs &a, cudaStream_t s);

}  // namespace moe

// Top-k routing of one token by one warp (used by the routing kernel and by
// the fused routing + permutation kernel).
//
// Method: "DeepSeek V4 Flash 单卡 MI300X" (txtmix.com) §一 — each token
// picks k of E experts (top-6 of 256) from its router scores; §三 — the
// routing bitmatrix (one bit per chosen expert). Selection runs on the fp32
// logits themselves (softmax is monotone); equal logits go to the lower
// expert index and -0.0 equals +0.0. Weights are the softmax restricted to
// the chosen experts and renormalised, i.e. exp(l_j - l_max) / sum over the
// chosen exp(l_i - l_max).
//
// Each lane owns experts lane, lane+32, ... (coalesced 128-byte loads) as
// order-preserving 32-bit keys. Every round takes the warp maximum key with
// redux.sync; a ballot finds the lanes holding it (one lane: its lowest value
// index with that key wins; several: the lowest expert index among them, by a
// second redux.sync).
#pragma once
#include <cstdint>

namespace moe {

// Order-preserving key of a finite float, with -0.0 folded onto +0.0.
__device__ __forceinline__ uint32_t float_key(float f)
{
    uint32_t u = __float_as_uint(f);
    if ((u << 1) == 0u) u = 0u;                 // -0.0 -> +0.0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Route token t (whole warp, converged). VPL = ceil(E / 32) values per lane. ids_copy (may be null):
// a second destination of the ids, e.g. shared memory for a permutation in the same block.
template <int VPL>
__device__ __forceinline__ void route_token(const float *__restrict__ logits, int t, int E, int k,
                                            int32_t *__restrict__ ids, float *__restrict__ w,
                                            uint32_t *__restrict__ bitmatrix, int32_t *ids_copy = nullptr)
{
    const uint32_t lane = threadIdx.x & 31u;
    const float *row = logits + (int64_t)t * E;
    uint32_t key[VPL];
#pragma unroll
    for (int v = 0; v < VPL; ++v) {
        int e = (int)lane + 32 * v;
        key[v] = (e < E) ? float_key(__ldg(row + e)) : 0u;   // values past E never win (k <= E)
    }
    // Chosen values get key 0, below every finite logit's key (>= 0x00800000), like lanes past E.
    int my_id = -1;               // lane j < k keeps the j-th choice
    float my_logit = 0.f;

    for (int j = 0; j < k; ++j) {
        uint32_t best = key[0];   // this lane's largest remaining key, at its lowest value index
        int best_v = 0;
#pragma unroll
        for (int v = 1; v < VPL; ++v) {
            const bool gt = key[v] > best;
            best = gt ? key[v] : best;
            best_v = gt ? v : best_v;
        }
        const uint32_t wmax = __reduce_max_sync(0xFFFFFFFFu, best);
        const unsigned holders = __ballot_sync(0xFFFFFFFFu, best == wmax);
        int win;
        if (__popc(holders) == 1) {                  // warp-uniform: the common case, no tie across lanes
            const int wl = __ffs(holders) - 1;
            win = wl + 32 * __shfl_sync(0xFFFFFFFFu, best_v, wl);
        } else {                                     // equal keys in several lanes: lowest expert index
            const uint32_t cand = best == wmax ? lane + 32u * (uint32_t)best_v : 0xFFFFFFFFu;
            win = (int)__reduce_min_sync(0xFFFFFFFFu, cand);
        }
        const bool mine = (win & 31) == (int)lane;
#pragma unroll
        for (int v = 0; v < VPL; ++v) key[v] = (mine && v == best_v) ? 0u : key[v];
        if ((int)lane == j) {
            my_id = win;
            my_logit = row[win];
        }
    }

    // softmax over the chosen k, shifted by the first (largest) logit
    float lmax = __shfl_sync(0xFFFFFFFFu, my_logit, 0);
    float ex = ((int)lane < k) ? expf(my_logit - lmax) : 0.f;
    float z = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
    if ((int)lane < k) {
        ids[(int64_t)t * k + lane] = my_id;
        w[(int64_t)t * k + lane] = ex / z;
        if (ids_copy) ids_copy[t * k + (int)lane] = my_id;
    }
    if (bitmatrix) {
        // every lane takes part in the shuffles; lane q builds word q (E <= 1024: at most 32 words)
        const int words = (E + 31) >> 5;
        uint32_t bits = 0u;
        for (int j = 0; j < k; ++j) {
            const int e = __shfl_sync(0xFFFFFFFFu, my_id, j);
            if ((e >> 5) == (int)lane) bits |= 1u << (e & 31);
        }
        if ((int)lane < words) bitmatrix[(int64_t)t * words + lane] = bits;
    }
}

}  // namespace moe

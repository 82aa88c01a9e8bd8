// Top-k expert routing: one warp per token (see route_token.cuh for the
// method and its citations).
#include <cstdint>

#include "moe_internal.h"
#include "route_token.cuh"

namespace moe {

template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, int T, int E, int k,
                                                     int32_t *__restrict__ ids, float *__restrict__ w,
                                                     uint32_t *__restrict__ bitmatrix)
{
    griddep_launch_dependents();      // the permutation launched next waits for this grid's ids
    const int warps = blockDim.x >> 5;
    const int t = blockIdx.x * warps + (threadIdx.x >> 5);
    if (t >= T) return;
    route_token<VPL>(logits, t, E, k, ids, w, bitmatrix);
}

cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                         uint32_t *bitmatrix, cudaStream_t s)
{
    const int threads = 256, per_block = threads / 32;
    const int blocks = (T + per_block - 1) / per_block;
    const int vpl = (E + 31) / 32;
    if (vpl <= 1) route_kernel<1><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w, bitmatrix);
    else if (vpl <= 2) route_kernel<2><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w, bitmatrix);
    else if (vpl <= 4) route_kernel<4><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w, bitmatrix);
    else if (vpl <= 8) route_kernel<8><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w, bitmatrix);
    else if (vpl <= 16) route_kernel<16><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w, bitmatrix);
    else route_kernel<32><<<blocks, threads, 0, s>>>(logits, T, E, k, ids, w, bitmatrix);
    note_launch(1);
    return cudaGetLastError();
}

}  // namespace moe

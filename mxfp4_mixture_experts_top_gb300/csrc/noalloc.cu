// moe_mxfp4_forward_noalloc: the layer forward with its scratch memory in a
// file-scope device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they run the layer — a runtime that forbids allocation after start-up, a
// plugin whose host framework owns the allocator and hands out no scratch
// space, or code that must not call cudaMalloc/cudaFree because they can
// synchronise the device. They still pass their inputs and outputs; only the
// intermediates (gathered activation terms, the MXFP8 terms of SiLU(gate)*up,
// per-pair W2 outputs) and the forward's device error word live in the array
// below.
//
// Cost: every GPU that loads this library holds MOE_NOALLOC_SCRATCH_BYTES of
// device memory until the process exits. Calls share the array: two calls
// whose work overlaps on the GPU (for example on two streams) race on it.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/moe_mxfp4.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[MOE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// cudaGetSymbolAddress once per device (with that device current) and cached.
moe_status_t scratch_on_current_device(void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status_t moe_mxfp4_forward_noalloc(const moe_layer_desc *desc, const uint16_t *d_x,
                                                  const void *d_packed, const float *d_topk_w,
                                                  const int32_t *d_offsets, const int32_t *d_padded_offsets,
                                                  const int32_t *d_row_to_pair, void *d_y, void *stream)
{
    size_t layout[7];
    const moe_status_t valid = moe_mxfp4_workspace_layout(desc, layout);   // same checks as the forward
    if (valid != MOE_OK) return valid;
    if (layout[6] > (size_t)MOE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;   // layer too large for the array
    void *scratch = nullptr;
    const moe_status_t st = scratch_on_current_device(&scratch);
    if (st != MOE_OK) return st;
    // The forward clears its own device error word and writes every other
    // scratch byte it later reads, so stale contents from earlier calls are harmless.
    return moe_mxfp4_forward(desc, d_x, d_packed, d_topk_w, d_offsets, d_padded_offsets, d_row_to_pair, d_y,
                             scratch, (size_t)MOE_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" moe_status_t moe_mxfp4_noalloc_read_device_error(int *code, void *stream)
{
    if (!code) return MOE_ERR_INVALID_ARG;
    void *scratch = nullptr;
    const moe_status_t st = scratch_on_current_device(&scratch);
    if (st != MOE_OK) return st;
    // the error word sits at offset 0 of the forward's workspace layout
    return moe_read_device_error(scratch, code, stream);
}

// adaln_out_bwd_noalloc: the LayerNorm/modulation backward for callers that
// cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc (or any allocator) at
// the point where they run the backward: a plugin inside an inference or
// training engine that owns every byte of device memory and forbids
// allocations inside its execute hook, a real-time loop that must never take
// the allocator's locks or risk its implicit device synchronisation, or code
// with a fixed memory budget decided at start-up.  For them this entry point
// takes no workspace: the token-tree partials live in a file-scope device
// array that is part of the library image.  Every GPU that loads the library
// holds this array (kNoAllocScratchBytes) until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "adaln.h"
#include "internal.h"

namespace adaln {

// 24 MiB: the workspace of adaln_out_bwd (the level-0 token-tree partials)
// for B = 2 and S <= 8192, or B = 1 and S <= 16384, at D = 3072.
constexpr size_t kNoAllocScratchBytes = 24u << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64];  // device address of the array, per device, once looked up

// The array's device address on the current device `dev`.  In host code the
// name g_noalloc_scratch is only a host-side stand-in, never a device address,
// so the address is asked from the runtime, with the device current.
adaln_status noalloc_scratch(int dev, void **ptr) {
    if (dev < 0 || dev >= 64) return ADALN_ERR_DEVICE;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return ADALN_ERR_CUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return ADALN_OK;
}

}  // namespace
}  // namespace adaln

extern "C" {

adaln_status adaln_out_bwd_noalloc(const adaln_bf16 *dy, const adaln_bf16 *x, const adaln_bf16 *emb,
                                   const float *mean, const float *rstd, adaln_bf16 *dx, float *d_emb, int B, int S,
                                   int D, void *stream) {
    using namespace adaln;
    // the checks of adaln_out_bwd, in its order: sizes (here also: the partials
    // must fit in the library's array), NULL pointers, alignment, overlaps,
    // then the device; only then the array's address
    adaln_status st = check_out_bwd_args(dy, x, emb, mean, rstd, dx, d_emb, B, S, D);
    if (st == ADALN_ERR_SHAPE) return st;
    if (adaln_out_bwd_workspace_bytes(B, S, D) > kNoAllocScratchBytes) return ADALN_ERR_SHAPE;
    if (st != ADALN_OK) return st;
    DeviceInfo dev;
    st = check_current_device(&dev);
    if (st != ADALN_OK) return st;
    void *scratch = nullptr;
    if (adaln_out_bwd_workspace_bytes(B, S, D) > 0) {
        st = noalloc_scratch(dev.device, &scratch);
        if (st != ADALN_OK) return st;
    }
    // the same kernels as adaln_out_bwd, with the array as workspace
    return adaln_out_bwd(dy, x, emb, mean, rstd, dx, d_emb, scratch, kNoAllocScratchBytes, B, S, D, stream);
}

}  // extern "C"

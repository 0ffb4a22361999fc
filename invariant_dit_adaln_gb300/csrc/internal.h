// Internal host-side interface between the C ABI (api.cu) and the kernel
// translation units (out.cu, proj.cu).  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "adaln.h"

namespace adaln {

struct DeviceInfo {
    int device;
    int sm_count;
    int cc_major;
    int cc_minor;
};

// api.cu: checks of the C ABI.  check_current_device: the current device and
// its properties; ADALN_ERR_DEVICE unless it is compute capability 10.3.
// check_out_bwd_args: the checks of adaln_out_bwd on its tensor arguments
// (sizes, NULL pointers, alignment, overlaps), the workspace excluded.
adaln_status check_current_device(DeviceInfo *info);
adaln_status check_out_bwd_args(const void *dy, const void *x, const void *emb, const float *mean, const float *rstd,
                                const void *dx, const float *d_emb, int B, int S, int D);

// Raise the dynamic shared-memory limit of a kernel once per (kernel, device).
cudaError_t ensure_smem_attr(const void *func, size_t bytes, const DeviceInfo &dev);

// Launch with programmatic dependent launch allowed: the kernel may start
// while the preceding kernel on the stream finishes; every kernel of this
// library calls griddepcontrol.wait before reading what a preceding kernel may
// write.  Every launch also asks for the largest shared-memory carve-out, so
// that consecutive kernels of the library never wait for an SM to change its
// L1/shared-memory split (which would also keep a dependent grid from starting
// early).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributePreferredSharedMemoryCarveout;
    attr[1].val.sharedMemCarveout = (unsigned)cudaSharedmemCarveoutMaxShared;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// out.cu
// keep_out: write out as evict-last in L2 (a fused projection reads it next)
cudaError_t launch_out_fwd(const uint16_t *x, const uint16_t *emb, uint16_t *out, float *mean, float *rstd,
                           int B, int S, int D, float eps, cudaStream_t stream, const DeviceInfo &dev,
                           bool keep_out = false);
// the block-level norm's forward fused into the LayerNorm kernel (D <= 4096)
bool out_fwd_res_supported(int D);
cudaError_t launch_out_fwd_res(const uint16_t *x, const uint16_t *residual, const uint16_t *gate,
                               const uint16_t *emb, uint16_t *r, uint16_t *out, float *mean, float *rstd, int B,
                               int S, int D, float eps, cudaStream_t stream, const DeviceInfo &dev);
// keep_dx: write dx as evict-last in L2 (a following kernel reads it)
cudaError_t launch_out_bwd(const uint16_t *dy, const uint16_t *x, const uint16_t *emb, const float *mean,
                           const float *rstd, uint16_t *dx, float *d_emb, void *ws, int B, int S, int D,
                           cudaStream_t stream, const DeviceInfo &dev,
                           bool keep_dx = false);
cudaError_t launch_token_tree(const float *in, float *out, void *ws, int B, int S, int H, cudaStream_t stream,
                              const DeviceInfo &dev);
int read_and_clear_device_error();
// the token tree's levels >= 1 from level-0 nodes sig, kap [B][T][H]; zero fill
cudaError_t launch_fold(const float *sig, const float *kap, float *out, int B, int T, int H, cudaStream_t stream,
                        const DeviceInfo &dev);
cudaError_t launch_zero(float *p, size_t n, cudaStream_t stream);

// f32.cu: the fp32 execution dtype (D <= 4096)
cudaError_t launch_f32_proj_fwd(const float *temb, const float *W, const float *bias, float *emb, float *u, int B,
                                int D, cudaStream_t stream, const DeviceInfo &dev);
cudaError_t launch_f32_out_fwd(const float *x, const float *emb, float *out, float *mean, float *rstd, int B, int S,
                               int D, float eps, cudaStream_t stream, const DeviceInfo &dev);
cudaError_t launch_f32_out_bwd(const float *dy, const float *x, const float *emb, const float *mean,
                               const float *rstd, float *dx, float *d_emb, void *ws, int B, int S, int D,
                               cudaStream_t stream, const DeviceInfo &dev);
size_t f32_proj_bwd_ws_bytes(int B, int D);
cudaError_t launch_f32_proj_bwd(const float *d_emb, const float *temb, const float *u, const float *W,
                                float *d_temb, float *dW_acc, float *db_acc, int accumulate, void *ws, int B, int D,
                                cudaStream_t stream, const DeviceInfo &dev);

// res.cu: the block-level modulated norm with a gated residual
cudaError_t launch_res_fwd(const uint16_t *x, const uint16_t *residual, const uint16_t *gate, const uint16_t *emb,
                           uint16_t *r, uint16_t *out, float *mean, float *rstd, int B, int S, int D, float eps,
                           cudaStream_t stream, const DeviceInfo &dev);
cudaError_t launch_res_bwd(const uint16_t *d_out, const uint16_t *d_r, const uint16_t *x, const uint16_t *r,
                           const uint16_t *gate, const uint16_t *emb, const float *mean, const float *rstd,
                           uint16_t *d_x, uint16_t *d_residual, float *d_emb, float *d_gate, void *ws, int B, int S,
                           int D, cudaStream_t stream, const DeviceInfo &dev);

// proj.cu
cudaError_t launch_proj_fwd(const uint16_t *temb, const uint16_t *W, const uint16_t *bias, uint16_t *emb,
                            uint16_t *u, int B, int D, cudaStream_t stream, const DeviceInfo &dev);
cudaError_t launch_proj_bwd(const float *d_emb, const uint16_t *temb, const uint16_t *u, const uint16_t *W,
                            uint16_t *d_temb, float *dW_acc, float *db_acc, uint16_t *dW, uint16_t *db,
                            int accumulate, void *ws, int B, int D, cudaStream_t stream, const DeviceInfo &dev);
int read_and_clear_proj_error();

// tc_proj.cu: emb = u W^T + bias on the tensor cores, for D a multiple of 64
// (and a driver that provides the tensor-map encoder); u written beforehand.
bool proj_fwd_tc_supported(int D);
int proj_fwd_tc_ksplit(int D);
cudaError_t launch_proj_fwd_tc(const uint16_t *u, const uint16_t *W, const uint16_t *bias, uint16_t *emb, int B,
                               int D, cudaStream_t stream, const DeviceInfo &dev);
int read_and_clear_tc_error();
// the LayerNorm forward, then y = out Wp^T + bp on the tensor cores (J = 64,
// D a multiple of 64)
bool proj_out_tc_supported(int D, int J);
cudaError_t launch_out_fwd_proj(const uint16_t *x, const uint16_t *emb, const uint16_t *Wp, const uint16_t *bp,
                                uint16_t *out, float *mean, float *rstd, uint16_t *y, int B, int S, int D,
                                float eps, cudaStream_t stream, const DeviceInfo &dev);
cudaError_t launch_wgrad_rows(const float *d_emb, const uint16_t *u, int n0, int n1, float *dW_acc, float *db_acc,
                              uint16_t *dW, uint16_t *db, int accumulate, int B, int D, cudaStream_t stream);

}  // namespace adaln

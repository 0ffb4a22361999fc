// C ABI of libadaln.so (declared in include/adaln.h): host-side argument
// checks, then the launches.  Every check runs before anything is enqueued;
// the order is shapes and argument values, NULL pointers (a pointer may be
// NULL only when its buffer has zero bytes), alignment, overlaps, workspace
// size, current device.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <unordered_map>

#include "adaln.h"
#include "common.cuh"
#include "internal.h"

namespace adaln {

namespace {

struct Buf {
    const void *p;
    size_t bytes;
};

bool overlaps(const Buf &a, const Buf &b) {
    if (!a.p || !b.p || a.bytes == 0 || b.bytes == 0) return false;
    const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
    return a0 < b0 + b.bytes && b0 < a0 + a.bytes;
}

// Every output against every input, every other output and the workspace.
bool any_alias(const Buf *outs, int nout, const Buf *ins, int nin) {
    for (int i = 0; i < nout; ++i) {
        for (int j = 0; j < nin; ++j)
            if (overlaps(outs[i], ins[j])) return true;
        for (int j = i + 1; j < nout; ++j)
            if (overlaps(outs[i], outs[j])) return true;
    }
    return false;
}

bool aligned16(const void *p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; }

// a buffer with bytes > 0 needs a pointer
bool missing(const Buf &b) { return b.bytes > 0 && b.p == nullptr; }
bool any_missing(const Buf *bufs, int n) {
    for (int i = 0; i < n; ++i)
        if (missing(bufs[i])) return true;
    return false;
}

bool valid_D(int D) { return D >= 8 && D <= kMaxD && D % 8 == 0; }

bool valid_BS(int B, int S, int D) {
    if (B < 0 || S < 0 || S > kMaxS || B > 65535) return false;
    return (long double)B * S * D < 1099511627776.0L;  // 2^40
}

size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

std::mutex g_mu;

// Current device, its SM count and compute capability, cached per device.
adaln_status current_device(DeviceInfo *info) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return ADALN_ERR_DEVICE;
    }
    static std::unordered_map<int, DeviceInfo> cache;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = cache.find(dev);
        if (it != cache.end()) {
            *info = it->second;
            return (info->cc_major == 10 && info->cc_minor == 3) ? ADALN_OK : ADALN_ERR_DEVICE;
        }
    }
    DeviceInfo d{dev, 0, 0, 0};
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return ADALN_ERR_DEVICE;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        cache[dev] = d;
    }
    *info = d;
    return (d.cc_major == 10 && d.cc_minor == 3) ? ADALN_OK : ADALN_ERR_DEVICE;
}

adaln_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return ADALN_OK;
    cudaGetLastError();  // clear a non-sticky launch error
    return ADALN_ERR_CUDA;
}

size_t tiles(int S) { return (size_t)((S + kTile - 1) / kTile); }

}  // namespace

adaln_status check_current_device(DeviceInfo *info) { return current_device(info); }

adaln_status check_out_bwd_args(const void *dy, const void *x, const void *emb, const float *mean, const float *rstd,
                                const void *dx, const float *d_emb, int B, int S, int D) {
    if (!valid_D(D) || !valid_BS(B, S, D)) return ADALN_ERR_SHAPE;
    const size_t rows = (size_t)B * S;
    const Buf ins[] = {{dy, rows * D * 2}, {x, rows * D * 2}, {emb, (size_t)B * 2 * D * 2}, {mean, rows * 4},
                       {rstd, rows * 4}};
    const Buf outs[] = {{dx, rows * D * 2}, {d_emb, (size_t)B * 2 * D * 4}};
    if (any_missing(ins, 5) || any_missing(outs, 2)) return ADALN_ERR_NULL;
    if (!aligned16(dy) || !aligned16(x) || !aligned16(emb) || !aligned16(mean) || !aligned16(rstd) ||
        !aligned16(dx) || !aligned16(d_emb))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 2, ins, 5)) return ADALN_ERR_ALIAS;
    return ADALN_OK;
}

cudaError_t ensure_smem_attr(const void *func, size_t bytes, const DeviceInfo &dev) {
    static std::unordered_map<const void *, size_t> done[64];
    const int slot = dev.device & 63;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        auto it = done[slot].find(func);
        if (it != done[slot].end() && it->second >= bytes) return cudaSuccess;
    }
    if (bytes <= 48 * 1024) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) {
        std::lock_guard<std::mutex> lk(g_mu);
        size_t &v = done[slot][func];
        if (bytes > v) v = bytes;
    }
    return e;
}

}  // namespace adaln

using namespace adaln;

extern "C" {

const char *adaln_status_string(int status) {
    switch (status) {
        case ADALN_OK: return "ADALN_OK";
        case ADALN_ERR_NULL: return "ADALN_ERR_NULL: a required pointer is NULL";
        case ADALN_ERR_SHAPE: return "ADALN_ERR_SHAPE: a size is out of range";
        case ADALN_ERR_ALIGN: return "ADALN_ERR_ALIGN: a pointer is not 16-byte aligned";
        case ADALN_ERR_ALIAS: return "ADALN_ERR_ALIAS: an output overlaps an input, another output or the workspace";
        case ADALN_ERR_WORKSPACE: return "ADALN_ERR_WORKSPACE: workspace missing or too small";
        case ADALN_ERR_DEVICE: return "ADALN_ERR_DEVICE: no current CUDA device, or it is not compute capability 10.3";
        case ADALN_ERR_CUDA: return "ADALN_ERR_CUDA: a CUDA call or kernel launch failed";
        case ADALN_ERR_ARG: return "ADALN_ERR_ARG: an argument value is invalid";
        default: return "unknown adaln status";
    }
}

int adaln_version(void) { return (1 << 16) | 0; }

size_t adaln_out_bwd_workspace_bytes(int B, int S, int D) {
    if (B <= 0 || S <= 0 || D <= 0) return 0;
    return round256(2 * (size_t)B * tiles(S) * 2 * (size_t)D * sizeof(float));
}

size_t token_sum_tree_workspace_bytes(int B, int S, int H) {
    if (B <= 0 || S <= 0 || H <= 0) return 0;
    return round256(2 * (size_t)B * tiles(S) * (size_t)H * sizeof(float));
}

size_t adaln_proj_bwd_workspace_bytes(int B, int D) {
    if (B <= 0 || D <= 0) return 0;
    const size_t nslab = (size_t)(2 * D + kProjSlabRows - 1) / kProjSlabRows;
    return round256(nslab * (size_t)B * D * sizeof(float));
}

adaln_status adaln_proj_fwd(const adaln_bf16 *temb, const adaln_bf16 *W, const adaln_bf16 *bias, adaln_bf16 *emb,
                            adaln_bf16 *u, int B, int D, void *stream) {
    if (!valid_D(D) || B < 0 || B > (1 << 20)) return ADALN_ERR_SHAPE;
    const size_t N = 2 * (size_t)D;
    const Buf ins[] = {{temb, (size_t)B * D * 2}, {W, N * D * 2}, {bias, N * 2}};
    const Buf outs[] = {{emb, (size_t)B * N * 2}, {u, (size_t)B * D * 2}};
    if (any_missing(ins, 3) || any_missing(outs, 2)) return ADALN_ERR_NULL;
    if (!aligned16(temb) || !aligned16(W) || !aligned16(bias) || !aligned16(emb) || !aligned16(u))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 2, ins, 3)) return ADALN_ERR_ALIAS;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (B == 0) return ADALN_OK;
    return from_cuda(launch_proj_fwd(temb, W, bias, emb, u, B, D, (cudaStream_t)stream, dev));
}

adaln_status adaln_out_fwd(const adaln_bf16 *x, const adaln_bf16 *emb, adaln_bf16 *out, float *mean, float *rstd,
                           int B, int S, int D, float eps, void *stream) {
    if (!valid_D(D) || !valid_BS(B, S, D)) return ADALN_ERR_SHAPE;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return ADALN_ERR_ARG;
    const size_t rows = (size_t)B * S;
    const Buf ins[] = {{x, rows * D * 2}, {emb, (size_t)B * 2 * D * 2}};
    const Buf outs[] = {{out, rows * D * 2}, {mean, rows * 4}, {rstd, rows * 4}};
    if (any_missing(ins, 2) || any_missing(outs, 3)) return ADALN_ERR_NULL;
    if (!aligned16(x) || !aligned16(emb) || !aligned16(out) || !aligned16(mean) || !aligned16(rstd))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 3, ins, 2)) return ADALN_ERR_ALIAS;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (rows == 0) return ADALN_OK;
    return from_cuda(launch_out_fwd(x, emb, out, mean, rstd, B, S, D, eps, (cudaStream_t)stream, dev));
}

adaln_status adaln_out_bwd(const adaln_bf16 *dy, const adaln_bf16 *x, const adaln_bf16 *emb, const float *mean,
                           const float *rstd, adaln_bf16 *dx, float *d_emb, void *workspace, size_t workspace_bytes,
                           int B, int S, int D, void *stream) {
    adaln_status chk = check_out_bwd_args(dy, x, emb, mean, rstd, dx, d_emb, B, S, D);
    if (chk == ADALN_ERR_SHAPE || chk == ADALN_ERR_NULL) return chk;
    const size_t rows = (size_t)B * S;
    const size_t need = adaln_out_bwd_workspace_bytes(B, S, D);
    if (chk == ADALN_ERR_ALIGN || !aligned16(workspace)) return ADALN_ERR_ALIGN;
    const Buf ins[] = {{dy, rows * D * 2}, {x, rows * D * 2}, {emb, (size_t)B * 2 * D * 2}, {mean, rows * 4},
                       {rstd, rows * 4}};
    const Buf outs[] = {{dx, rows * D * 2}, {d_emb, (size_t)B * 2 * D * 4}, {workspace, need}};
    if (chk == ADALN_ERR_ALIAS || any_alias(outs, 3, ins, 5)) return ADALN_ERR_ALIAS;
    if (need > 0 && (!workspace || workspace_bytes < need)) return ADALN_ERR_WORKSPACE;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (B == 0) return ADALN_OK;
    return from_cuda(launch_out_bwd(dy, x, emb, mean, rstd, dx, d_emb, workspace, B, S, D, (cudaStream_t)stream, dev));
}

adaln_status token_sum_tree(const float *in, float *out, int B, int S, int H, void *workspace, size_t workspace_bytes,
                            void *stream) {
    if (H < 4 || H > (1 << 20) || H % 4 != 0 || B < 0 || B > 65535 || S < 0 || S > kMaxS ||
        (long double)B * S * H >= 1099511627776.0L)
        return ADALN_ERR_SHAPE;
    const size_t need = token_sum_tree_workspace_bytes(B, S, H);
    const Buf ins[] = {{in, (size_t)B * S * H * 4}};
    const Buf outs[] = {{out, (size_t)B * H * 4}, {workspace, need}};
    if (any_missing(ins, 1) || any_missing(outs, 1)) return ADALN_ERR_NULL;
    if (!aligned16(in) || !aligned16(out) || !aligned16(workspace)) return ADALN_ERR_ALIGN;
    if (any_alias(outs, 2, ins, 1)) return ADALN_ERR_ALIAS;
    if (need > 0 && (!workspace || workspace_bytes < need)) return ADALN_ERR_WORKSPACE;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (B == 0) return ADALN_OK;
    return from_cuda(launch_token_tree(in, out, workspace, B, S, H, (cudaStream_t)stream, dev));
}

adaln_status adaln_out_fwd_proj(const adaln_bf16 *x, const adaln_bf16 *emb, const adaln_bf16 *Wp,
                                const adaln_bf16 *bp, adaln_bf16 *out, float *mean, float *rstd, adaln_bf16 *y,
                                int B, int S, int D, int J, float eps, void *stream) {
    if (!valid_D(D) || D % 64 != 0 || J != 64 || !valid_BS(B, S, D) || (long long)B * S > 65535LL * 128)
        return ADALN_ERR_SHAPE;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return ADALN_ERR_ARG;
    const size_t rows = (size_t)B * S;
    const Buf ins[] = {{x, rows * D * 2}, {emb, (size_t)B * 2 * D * 2}, {Wp, (size_t)J * D * 2}, {bp, (size_t)J * 2}};
    const Buf outs[] = {{out, rows * D * 2}, {mean, rows * 4}, {rstd, rows * 4}, {y, rows * J * 2}};
    if (any_missing(ins, 4) || any_missing(outs, 4)) return ADALN_ERR_NULL;
    if (!aligned16(x) || !aligned16(emb) || !aligned16(Wp) || !aligned16(bp) || !aligned16(out) ||
        !aligned16(mean) || !aligned16(rstd) || !aligned16(y))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 4, ins, 4)) return ADALN_ERR_ALIAS;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (rows == 0) return ADALN_OK;
    if (!proj_out_tc_supported(D, J)) return ADALN_ERR_CUDA;  // the driver offers no tensor-map encoder
    return from_cuda(launch_out_fwd_proj(x, emb, Wp, bp, out, mean, rstd, y, B, S, D, eps, (cudaStream_t)stream, dev));
}

// ---- fp32 execution dtype (D <= 4096) ----

adaln_status adaln_f32_proj_fwd(const float *temb, const float *W, const float *bias, float *emb, float *u, int B,
                                int D, void *stream) {
    if (!valid_D(D) || D > 4096 || B < 0 || B > (1 << 20)) return ADALN_ERR_SHAPE;
    const size_t N = 2 * (size_t)D;
    const Buf ins[] = {{temb, (size_t)B * D * 4}, {W, N * D * 4}, {bias, N * 4}};
    const Buf outs[] = {{emb, (size_t)B * N * 4}, {u, (size_t)B * D * 4}};
    if (any_missing(ins, 3) || any_missing(outs, 2)) return ADALN_ERR_NULL;
    if (!aligned16(temb) || !aligned16(W) || !aligned16(bias) || !aligned16(emb) || !aligned16(u))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 2, ins, 3)) return ADALN_ERR_ALIAS;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (B == 0) return ADALN_OK;
    return from_cuda(launch_f32_proj_fwd(temb, W, bias, emb, u, B, D, (cudaStream_t)stream, dev));
}

adaln_status adaln_f32_out_fwd(const float *x, const float *emb, float *out, float *mean, float *rstd, int B, int S,
                               int D, float eps, void *stream) {
    if (!valid_D(D) || D > 4096 || !valid_BS(B, S, D)) return ADALN_ERR_SHAPE;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return ADALN_ERR_ARG;
    const size_t rows = (size_t)B * S;
    const Buf ins[] = {{x, rows * D * 4}, {emb, (size_t)B * 2 * D * 4}};
    const Buf outs[] = {{out, rows * D * 4}, {mean, rows * 4}, {rstd, rows * 4}};
    if (any_missing(ins, 2) || any_missing(outs, 3)) return ADALN_ERR_NULL;
    if (!aligned16(x) || !aligned16(emb) || !aligned16(out) || !aligned16(mean) || !aligned16(rstd))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 3, ins, 2)) return ADALN_ERR_ALIAS;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (rows == 0) return ADALN_OK;
    return from_cuda(launch_f32_out_fwd(x, emb, out, mean, rstd, B, S, D, eps, (cudaStream_t)stream, dev));
}

size_t adaln_f32_out_bwd_workspace_bytes(int B, int S, int D) { return adaln_out_bwd_workspace_bytes(B, S, D); }

adaln_status adaln_f32_out_bwd(const float *dy, const float *x, const float *emb, const float *mean,
                               const float *rstd, float *dx, float *d_emb, void *workspace, size_t workspace_bytes,
                               int B, int S, int D, void *stream) {
    if (!valid_D(D) || D > 4096 || !valid_BS(B, S, D)) return ADALN_ERR_SHAPE;
    const size_t rows = (size_t)B * S;
    const size_t need = adaln_f32_out_bwd_workspace_bytes(B, S, D);
    const Buf ins[] = {{dy, rows * D * 4}, {x, rows * D * 4}, {emb, (size_t)B * 2 * D * 4}, {mean, rows * 4},
                       {rstd, rows * 4}};
    const Buf outs[] = {{dx, rows * D * 4}, {d_emb, (size_t)B * 2 * D * 4}, {workspace, need}};
    if (any_missing(ins, 5) || any_missing(outs, 2)) return ADALN_ERR_NULL;
    if (!aligned16(dy) || !aligned16(x) || !aligned16(emb) || !aligned16(mean) || !aligned16(rstd) ||
        !aligned16(dx) || !aligned16(d_emb) || !aligned16(workspace))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 3, ins, 5)) return ADALN_ERR_ALIAS;
    if (need > 0 && (!workspace || workspace_bytes < need)) return ADALN_ERR_WORKSPACE;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (B == 0) return ADALN_OK;
    return from_cuda(launch_f32_out_bwd(dy, x, emb, mean, rstd, dx, d_emb, workspace, B, S, D, (cudaStream_t)stream,
                                        dev));
}

size_t adaln_f32_proj_bwd_workspace_bytes(int B, int D) {
    if (B <= 0 || D <= 0) return 0;
    return round256(f32_proj_bwd_ws_bytes(B, D));
}

adaln_status adaln_f32_proj_bwd(const float *d_emb, const float *temb, const float *u, const float *W, float *d_temb,
                                float *dW_acc, float *db_acc, int accumulate, void *workspace,
                                size_t workspace_bytes, int B, int D, void *stream) {
    if (!valid_D(D) || D > 4096 || B < 0 || B > (1 << 20)) return ADALN_ERR_SHAPE;
    if (accumulate != 0 && accumulate != 1) return ADALN_ERR_ARG;
    const size_t N = 2 * (size_t)D;
    const size_t need = adaln_f32_proj_bwd_workspace_bytes(B, D);
    const Buf ins[] = {{d_emb, (size_t)B * N * 4}, {temb, (size_t)B * D * 4}, {u, (size_t)B * D * 4},
                       {W, N * D * 4}};
    const Buf outs[] = {{d_temb, (size_t)B * D * 4}, {dW_acc, dW_acc ? N * D * 4 : 0},
                        {db_acc, db_acc ? N * 4 : 0}, {workspace, need}};
    if (any_missing(ins, 4) || any_missing(outs, 1)) return ADALN_ERR_NULL;
    if (!aligned16(d_emb) || !aligned16(temb) || !aligned16(u) || !aligned16(W) || !aligned16(d_temb) ||
        !aligned16(dW_acc) || !aligned16(db_acc) || !aligned16(workspace))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 4, ins, 4)) return ADALN_ERR_ALIAS;
    if (need > 0 && (!workspace || workspace_bytes < need)) return ADALN_ERR_WORKSPACE;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (B == 0) {
        // no samples: the gradient is its starting value (+0 unless accumulating)
        if (!accumulate) {
            cudaError_t e = cudaSuccess;
            if (dW_acc) e = cudaMemsetAsync(dW_acc, 0, N * D * 4, (cudaStream_t)stream);
            if (e == cudaSuccess && db_acc) e = cudaMemsetAsync(db_acc, 0, N * 4, (cudaStream_t)stream);
            return from_cuda(e);
        }
        return ADALN_OK;
    }
    return from_cuda(launch_f32_proj_bwd(d_emb, temb, u, W, d_temb, dW_acc, db_acc, accumulate, workspace, B, D,
                                         (cudaStream_t)stream, dev));
}

size_t adaln_scale_residual_norm_bwd_workspace_bytes(int B, int S, int D) {
    // the LayerNorm backward's tree nodes (2D columns), then the gate's (D
    // columns) in the same space
    return adaln_out_bwd_workspace_bytes(B, S, D);
}

adaln_status adaln_scale_residual_norm_fwd(const adaln_bf16 *x, const adaln_bf16 *residual, const adaln_bf16 *gate,
                                           const adaln_bf16 *emb, adaln_bf16 *r, adaln_bf16 *out, float *mean,
                                           float *rstd, int B, int S, int D, float eps, void *stream) {
    if (!valid_D(D) || !valid_BS(B, S, D)) return ADALN_ERR_SHAPE;
    if (!(eps >= 0.0f) || eps > 3.0e38f) return ADALN_ERR_ARG;
    const size_t rows = (size_t)B * S;
    const Buf ins[] = {{x, rows * D * 2}, {residual, rows * D * 2}, {gate, (size_t)B * D * 2},
                       {emb, (size_t)B * 2 * D * 2}};
    const Buf outs[] = {{r, rows * D * 2}, {out, rows * D * 2}, {mean, rows * 4}, {rstd, rows * 4}};
    if (any_missing(ins, 4) || any_missing(outs, 4)) return ADALN_ERR_NULL;
    if (!aligned16(x) || !aligned16(residual) || !aligned16(gate) || !aligned16(emb) || !aligned16(r) ||
        !aligned16(out) || !aligned16(mean) || !aligned16(rstd))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 4, ins, 4)) return ADALN_ERR_ALIAS;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (rows == 0) return ADALN_OK;
    return from_cuda(launch_res_fwd(x, residual, gate, emb, r, out, mean, rstd, B, S, D, eps, (cudaStream_t)stream,
                                    dev));
}

adaln_status adaln_scale_residual_norm_bwd(const adaln_bf16 *d_out, const adaln_bf16 *d_r, const adaln_bf16 *x,
                                           const adaln_bf16 *r, const adaln_bf16 *gate, const adaln_bf16 *emb,
                                           const float *mean, const float *rstd, adaln_bf16 *d_x,
                                           adaln_bf16 *d_residual, float *d_emb, float *d_gate, void *workspace,
                                           size_t workspace_bytes, int B, int S, int D, void *stream) {
    if (!valid_D(D) || !valid_BS(B, S, D)) return ADALN_ERR_SHAPE;
    const size_t rows = (size_t)B * S;
    const size_t need = adaln_scale_residual_norm_bwd_workspace_bytes(B, S, D);
    const Buf ins[] = {{d_out, rows * D * 2}, {x, rows * D * 2}, {r, rows * D * 2}, {gate, (size_t)B * D * 2},
                       {emb, (size_t)B * 2 * D * 2}, {mean, rows * 4}, {rstd, rows * 4},
                       {d_r, d_r ? rows * D * 2 : 0}};
    const Buf outs[] = {{d_x, rows * D * 2}, {d_residual, rows * D * 2}, {d_emb, (size_t)B * 2 * D * 4},
                        {d_gate, (size_t)B * D * 4}, {workspace, need}};
    if (any_missing(ins, 7) || any_missing(outs, 4)) return ADALN_ERR_NULL;
    if (!aligned16(d_out) || !aligned16(d_r) || !aligned16(x) || !aligned16(r) || !aligned16(gate) ||
        !aligned16(emb) || !aligned16(mean) || !aligned16(rstd) || !aligned16(d_x) || !aligned16(d_residual) ||
        !aligned16(d_emb) || !aligned16(d_gate) || !aligned16(workspace))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 5, ins, 8)) return ADALN_ERR_ALIAS;
    if (need > 0 && (!workspace || workspace_bytes < need)) return ADALN_ERR_WORKSPACE;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (B == 0) return ADALN_OK;
    return from_cuda(launch_res_bwd(d_out, d_r, x, r, gate, emb, mean, rstd, d_x, d_residual, d_emb, d_gate,
                                    workspace, B, S, D, (cudaStream_t)stream, dev));
}

adaln_status adaln_proj_bwd(const float *d_emb, const adaln_bf16 *temb, const adaln_bf16 *u, const adaln_bf16 *W,
                            adaln_bf16 *d_temb, float *dW_acc, float *db_acc, adaln_bf16 *dW, adaln_bf16 *db,
                            int accumulate, void *workspace, size_t workspace_bytes, int B, int D, void *stream) {
    if (!valid_D(D) || B < 0 || B > (1 << 20)) return ADALN_ERR_SHAPE;
    if (accumulate != 0 && accumulate != 1) return ADALN_ERR_ARG;
    const bool want_w = dW_acc || dW, want_b = db_acc || db;
    if (accumulate && ((want_w && !dW_acc) || (want_b && !db_acc))) return ADALN_ERR_ARG;
    const size_t N = 2 * (size_t)D;
    const size_t need = adaln_proj_bwd_workspace_bytes(B, D);
    const Buf ins[] = {{d_emb, (size_t)B * N * 4}, {temb, (size_t)B * D * 2}, {u, (size_t)B * D * 2},
                       {W, B > 0 ? N * D * 2 : 0}};
    // dW_acc / db_acc are read as well as written: they count as outputs here
    const Buf outs[] = {{d_temb, (size_t)B * D * 2}, {dW_acc, N * D * 4}, {db_acc, N * 4}, {dW, N * D * 2},
                        {db, N * 2}, {workspace, need}};
    if (any_missing(ins, 4) || missing(outs[0])) return ADALN_ERR_NULL;
    if (!aligned16(d_emb) || !aligned16(temb) || !aligned16(u) || !aligned16(W) || !aligned16(d_temb) ||
        !aligned16(dW_acc) || !aligned16(db_acc) || !aligned16(dW) || !aligned16(db) || !aligned16(workspace))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 6, ins, 4)) return ADALN_ERR_ALIAS;
    if (need > 0 && (!workspace || workspace_bytes < need)) return ADALN_ERR_WORKSPACE;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (B == 0 && !want_w && !want_b) return ADALN_OK;
    return from_cuda(launch_proj_bwd(d_emb, temb, u, W, d_temb, dW_acc, db_acc, dW, db, accumulate, workspace, B, D,
                                     (cudaStream_t)stream, dev));
}

adaln_status adaln_proj_wgrad_rows(const float *d_emb, const adaln_bf16 *u, int n0, int n1, float *dW_acc,
                                   float *db_acc, adaln_bf16 *dW, adaln_bf16 *db, int accumulate, int B, int D,
                                   void *stream) {
    if (!valid_D(D) || B < 0 || B > (1 << 20) || n0 < 0 || n1 < n0 || n1 > 2 * D) return ADALN_ERR_SHAPE;
    if (accumulate != 0 && accumulate != 1) return ADALN_ERR_ARG;
    const bool want_w = dW_acc || dW, want_b = db_acc || db;
    if (accumulate && ((want_w && !dW_acc) || (want_b && !db_acc))) return ADALN_ERR_ARG;
    const size_t N = 2 * (size_t)D, R = (size_t)(n1 - n0);
    const Buf ins[] = {{d_emb, (size_t)B * N * 4}, {u, (size_t)B * D * 2}};
    const Buf outs[] = {{dW_acc, R * D * 4}, {db_acc, R * 4}, {dW, R * D * 2}, {db, R * 2}};
    if (any_missing(ins, 2)) return ADALN_ERR_NULL;
    if (!aligned16(d_emb) || !aligned16(u) || !aligned16(dW_acc) || !aligned16(db_acc) || !aligned16(dW) ||
        !aligned16(db))
        return ADALN_ERR_ALIGN;
    if (any_alias(outs, 4, ins, 2)) return ADALN_ERR_ALIAS;
    DeviceInfo dev;
    adaln_status st = current_device(&dev);
    if (st != ADALN_OK) return st;
    if (R == 0 || (!want_w && !want_b)) return ADALN_OK;
    return from_cuda(launch_wgrad_rows(d_emb, u, n0, n1, dW_acc, db_acc, dW, db, accumulate, B, D,
                                       (cudaStream_t)stream));
}

int adaln_device_error(void) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    // the first kernel code of the LayerNorm kernels' word, then the projection
    // kernels' words; the drain bit of any word; all words cleared
    const int a = read_and_clear_device_error();
    const int b = read_and_clear_proj_error();
    const int c = read_and_clear_tc_error();
    if (a < 0 || b < 0 || c < 0) return -1;
    const int drain = (a | b | c) & (int)kErrDrainFailed;
    const int ca = a & ~(int)kErrDrainFailed, cb = b & ~(int)kErrDrainFailed, cc = c & ~(int)kErrDrainFailed;
    return (ca != 0 ? ca : cb != 0 ? cb : cc) | drain;
}

}  // extern "C"

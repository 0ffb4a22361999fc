// Block-level modulated norm with a gated residual (ScaleResidualLayerNorm-
// ScaleShift): the norm1/norm2 sites of every transformer block, with the
// rounding points of the final norm (miles_diffusion PR 108, Summary, root
// cause 1, and "Patches": fp32 LayerNorm, bf16 (1 + scale), fp32 modulation;
// the residual stream's gated add runs in eager bf16, each operation computed
// in fp32 and rounded once to bf16).
//
//   forward:   r   = bf16(residual + bf16(gate * x))      gate [B, D], per sample
//              out = the LayerNorm + modulation of r       (out.cu, unchanged)
//   backward:  dr_ln, d_emb = the LayerNorm + modulation backward at r (out.cu)
//              gr         = bf16(dr_ln + d_r)             (r's two uses)
//              d_residual = gr,  d_x = bf16(gr * gate)
//              d_gate     = the token sum of bf16(gr * x), by the same fixed
//                           32-way tree as d_scale and d_shift
//
// The gated add and the backward's tail are elementwise per token (no
// reduction over d), so every token row is computed alone; the only reduction
// over tokens is d_gate's, through the tree, whose shape depends on S alone.
#include "common.cuh"
#include "internal.h"

namespace adaln {

// --------------------------------------------------------------------------
// forward: r = bf16(residual + bf16(gate * x)), 8 elements per thread and
// step, grid-stride; r keeps the default L2 policy, because the LayerNorm
// kernel reads it next.
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(256)
res_add_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ residual, const uint16_t *__restrict__ gate,
               uint16_t *__restrict__ r, long long n8, int S, int D) {
    pdl_wait();  // inputs may come from the preceding kernel
    const uint64_t pol = l2_evict_first();
    const long long V = D / 8;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (long long)gridDim.x * blockDim.x) {
        const long long row = i / V;
        const long long b = row / S;
        const int v = (int)(i - row * V);
        const uint4 xv = ldg16_hint(x + i * 8, pol);
        const uint4 rv = ldg16_hint(residual + i * 8, pol);
        const uint4 gv = ldg16(gate + b * D + (size_t)v * 8);
        const uint32_t xa[4] = {xv.x, xv.y, xv.z, xv.w}, ra[4] = {rv.x, rv.y, rv.z, rv.w},
                       ga[4] = {gv.x, gv.y, gv.z, gv.w};
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float lo = eager_add(bf16lo(ra[q]), eager_mul(bf16lo(ga[q]), bf16lo(xa[q])));
            const float hi = eager_add(bf16hi(ra[q]), eager_mul(bf16hi(ga[q]), bf16hi(xa[q])));
            o[q] = pack_bf16x2(lo, hi);
        }
        stg16(r + i * 8, make_uint4(o[0], o[1], o[2], o[3]));
    }
    pdl_trigger();
}

// --------------------------------------------------------------------------
// backward's tail: one thread per 8 columns of one (sample, 32-token tile);
// tokens in ascending order, four rows' loads in flight.  d_residual holds
// dr_ln on entry (written by the LayerNorm backward) and gr on exit.  The
// level-0 node of each column is the TwoSum (Neumaier) sum of the tile's
// products from (+0, +0), as in the LayerNorm backward's tiles.  Arithmetic on
// column pairs in packed fp32x2 instructions with explicit rounding; each
// eager bf16 operation is the fp32 result rounded once (round to nearest even).
// --------------------------------------------------------------------------
constexpr int kResRows = 4;

__global__ void __launch_bounds__(128)
res_gate_bwd_kernel(uint16_t *__restrict__ d_residual, const uint16_t *__restrict__ d_r,
                    const uint16_t *__restrict__ x, const uint16_t *__restrict__ gate, uint16_t *__restrict__ d_x,
                    float *__restrict__ ws_sig, float *__restrict__ ws_kap, int S, int D, int T) {
    const int V = D / 8;
    const int v = blockIdx.x * blockDim.x + threadIdx.x;
    const int t = blockIdx.y;
    const int b = blockIdx.z;
    pdl_wait();  // dr_ln comes from the preceding kernels; the workspace is free once they are done
    pdl_trigger();
    if (v >= V) return;
    const uint64_t pol = l2_evict_first();
    const int s0 = t * kTile;
    const int n = min(kTile, S - s0);
    const size_t base = ((size_t)b * S + s0) * D + (size_t)v * 8;
    // the sample's gate of this thread's columns, by column pair
    px2 gf[4];
    {
        const uint4 gv = ldg16(gate + (size_t)b * D + (size_t)v * 8);
        gf[0] = px_bf16(gv.x), gf[1] = px_bf16(gv.y), gf[2] = px_bf16(gv.z), gf[3] = px_bf16(gv.w);
    }
    // tree nodes of the gate products, by column pair, from (+0, +0)
    px2 sg[4], kp[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) sg[q] = kp[q] = 0ull;
    for (int i0 = 0; i0 < n; i0 += kResRows) {
        uint4 lv[kResRows], dv[kResRows], xv[kResRows];
#pragma unroll
        for (int k = 0; k < kResRows; ++k) {
            if (i0 + k < n) {
                const size_t o = base + (size_t)(i0 + k) * D;
                lv[k] = *reinterpret_cast<const uint4 *>(d_residual + o);
                dv[k] = d_r ? ldg16_hint(d_r + o, pol) : make_uint4(0u, 0u, 0u, 0u);
                xv[k] = ldg16_hint(x + o, pol);
            }
        }
#pragma unroll
        for (int k = 0; k < kResRows; ++k) {
            if (i0 + k < n) {
                const size_t o = base + (size_t)(i0 + k) * D;
                const uint32_t la[4] = {lv[k].x, lv[k].y, lv[k].z, lv[k].w};
                const uint32_t da[4] = {dv[k].x, dv[k].y, dv[k].z, dv[k].w};
                const uint32_t xa[4] = {xv[k].x, xv[k].y, xv[k].z, xv[k].w};
                uint32_t go[4], xo[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // gr = bf16(dr_ln + d_r) (exact bf16 values, so its store is exact)
                    const uint32_t grw = d_r ? px_to_bf16x2(px_add(px_bf16(la[q]), px_bf16(da[q]))) : la[q];
                    const px2 gr = px_bf16(grw);
                    go[q] = grw;
                    xo[q] = px_to_bf16x2(px_mul(gr, gf[q]));  // d_x = bf16(gr * gate)
                    // the tree product bf16(gr * x), by TwoSum
                    px_twosum(sg[q], kp[q], px_bf16(px_to_bf16x2(px_mul(gr, px_bf16(xa[q])))));
                }
                stg16_hint(d_residual + o, make_uint4(go[0], go[1], go[2], go[3]), pol);
                stg16_hint(d_x + o, make_uint4(xo[0], xo[1], xo[2], xo[3]), pol);
            }
        }
    }
    const size_t node = ((size_t)b * T + t) * D + (size_t)v * 8;
    stg16f(ws_sig + node, make_float4(px_lo(sg[0]), px_hi(sg[0]), px_lo(sg[1]), px_hi(sg[1])));
    stg16f(ws_sig + node + 4, make_float4(px_lo(sg[2]), px_hi(sg[2]), px_lo(sg[3]), px_hi(sg[3])));
    stg16f(ws_kap + node, make_float4(px_lo(kp[0]), px_hi(kp[0]), px_lo(kp[1]), px_hi(kp[1])));
    stg16f(ws_kap + node + 4, make_float4(px_lo(kp[2]), px_hi(kp[2]), px_lo(kp[3]), px_hi(kp[3])));
}

// --------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------
cudaError_t launch_res_fwd(const uint16_t *x, const uint16_t *residual, const uint16_t *gate, const uint16_t *emb,
                           uint16_t *r, uint16_t *out, float *mean, float *rstd, int B, int S, int D, float eps,
                           cudaStream_t stream, const DeviceInfo &dev) {
    const long long n8 = (long long)B * S * D / 8;
    long long grid = (n8 + 255) / 256;
    const long long cap = (long long)dev.sm_count * 8;
    if (grid > cap) grid = cap;
    if (out_fwd_res_supported(D))  // one kernel: r is formed, written and normalised in registers
        return launch_out_fwd_res(x, residual, gate, emb, r, out, mean, rstd, B, S, D, eps, stream, dev);
    cudaError_t err = launch_pdl(res_add_kernel, dim3((unsigned)grid), dim3(256), 0, stream, x, residual, gate, r,
                                 n8, S, D);
    if (err != cudaSuccess) return err;
    return launch_out_fwd(r, emb, out, mean, rstd, B, S, D, eps, stream, dev);
}

cudaError_t launch_res_bwd(const uint16_t *d_out, const uint16_t *d_r, const uint16_t *x, const uint16_t *r,
                           const uint16_t *gate, const uint16_t *emb, const float *mean, const float *rstd,
                           uint16_t *d_x, uint16_t *d_residual, float *d_emb, float *d_gate, void *ws, int B, int S,
                           int D, cudaStream_t stream, const DeviceInfo &dev) {
    // the LayerNorm + modulation backward at r: dr_ln into d_residual, d_emb
    // dr_ln stays in L2 for the tail kernel
    cudaError_t err = launch_out_bwd(d_out, r, emb, mean, rstd, d_residual, d_emb, ws, B, S, D, stream, dev, true);
    if (err != cudaSuccess) return err;
    if (S == 0) return launch_zero(d_gate, (size_t)B * D, stream);
    const int T = (S + kTile - 1) / kTile;
    float *sig = static_cast<float *>(ws);
    float *kap = sig + (size_t)B * T * D;
    const int V = D / 8;
    err = launch_pdl(res_gate_bwd_kernel, dim3((unsigned)((V + 127) / 128), (unsigned)T, (unsigned)B), dim3(128), 0,
                     stream, d_residual, d_r, x, gate, d_x, sig, kap, S, D, T);
    if (err != cudaSuccess) return err;
    return launch_fold(sig, kap, d_gate, B, T, D, stream, dev);
}

}  // namespace adaln

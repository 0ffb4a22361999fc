// The operator in the fp32 execution dtype (RL-Kernel PR 538 "Results": the
// FP32 timings and the BF16/FP32 acceptance gates): fp32 x, temb, W, bias, dy
// and fp32 outputs, no bf16 rounding anywhere, every step one fp32 rounding
// (no TF32: the tensor cores are not used).  The token trees and the weight
// gradient's sequential order are the bf16 path's.
//
//   u      = fp32(silu(t))                     (fp64, rounded once)
//   emb    = fp32 sum_k u W + bias             (fixed order: below)
//   mean, rstd, xhat = fp32(fp32(x - mean) * rstd)
//   out    = fp32(fp32(xhat * onep) + shift),  onep = fp32(1 + scale)
//   dx     = rstd * (gh - c1 - xhat * c2),     gh = fp32(g * onep), g = dy
//   d_emb  = the 32-way token trees of fp32(g * xhat) and g
//   d_temb = fp32(d_silu * silu'(t)),          d_silu = sum_n e W, e = d_emb
//   dW     = fma over samples ascending,        db = sum over samples ascending
#include "common.cuh"
#include "internal.h"

namespace adaln {

constexpr int kF32MaxD = 4096;  // the fp32 variant's largest row (a row per warp in registers)

__device__ __forceinline__ float4 ldf4_hint(const float *p, uint64_t pol) {
    const uint4 v = ldg16_hint(p, pol);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}

// --------------------------------------------------------------------------
// u = fp32(t / (1 + exp(-t))), computed in fp64 (B * D values)
// --------------------------------------------------------------------------
__global__ void __launch_bounds__(256) f32_silu_kernel(const float *__restrict__ t, float *__restrict__ u, long long n) {
    pdl_wait();
    pdl_trigger();
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        const double x = (double)t[i];
        u[i] = (float)(x * (1.0 / (1.0 + exp(-x))));
    }
}

// --------------------------------------------------------------------------
// emb[b,n] = sum_k u[b,k] W[n,k] + bias[n]: one warp per output row n; lane l
// takes the float4 vectors l, l + 32, ... of the row in ascending order, the
// four elements in order, one fused multiply-add each into one accumulator
// per sample; then a fixed xor butterfly over the lanes and the bias in fp32.
// The order depends on D only.  Samples in chunks of kF32BC (u of the chunk in
// shared memory; W is read again for every chunk).
// --------------------------------------------------------------------------
constexpr int kF32BC = 4;

__global__ void __launch_bounds__(256)
f32_proj_fwd_kernel(const float *__restrict__ u, const float *__restrict__ W, const float *__restrict__ bias,
                    float *__restrict__ emb, int B, int D) {
    extern __shared__ __align__(16) float us_f32[];  // [kF32BC][D]
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = 2 * D;
    const int n = blockIdx.x * 8 + warp;
    const bool live = n < N;
    const int V = D / 4;
    const float4 *wrow = reinterpret_cast<const float4 *>(W + (size_t)(live ? n : 0) * D);
    pdl_wait();
    pdl_trigger();
    for (int b0 = 0; b0 < B; b0 += kF32BC) {
        const int nb = min(kF32BC, B - b0);
        __syncthreads();
        for (int i = threadIdx.x; i < nb * V; i += blockDim.x)
            reinterpret_cast<float4 *>(us_f32)[i] = reinterpret_cast<const float4 *>(u + (size_t)b0 * D)[i];
        __syncthreads();
        float acc[kF32BC];
#pragma unroll
        for (int b = 0; b < kF32BC; ++b) acc[b] = 0.0f;
        for (int v0 = 0; v0 < V; v0 += 32 * 8) {
            float4 w[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int v = v0 + lane + 32 * j;
                w[j] = v < V ? __ldg(wrow + v) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int v = v0 + lane + 32 * j;
                if (v < V) {
#pragma unroll
                    for (int b = 0; b < kF32BC; ++b) {
                        if (b < nb) {
                            const float4 x = reinterpret_cast<const float4 *>(us_f32 + (size_t)b * D)[v];
                            acc[b] = __fmaf_rn(x.x, w[j].x, acc[b]);
                            acc[b] = __fmaf_rn(x.y, w[j].y, acc[b]);
                            acc[b] = __fmaf_rn(x.z, w[j].z, acc[b]);
                            acc[b] = __fmaf_rn(x.w, w[j].w, acc[b]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int b = 0; b < kF32BC; ++b) {
            if (b < nb) {
                const float tot = warp_sum(acc[b]);
                if (lane == 0 && live) emb[(size_t)(b0 + b) * N + n] = __fadd_rn(tot, bias[n]);
            }
        }
    }
}

// --------------------------------------------------------------------------
// LayerNorm + modulation forward: one warp per token row, rows of one sample
// per CTA (onep and shift of the sample in shared memory).  Lane l holds the
// float4 vectors l, l + 32, ... of the row in registers (D <= 4096).  Sums:
// per lane in vector order, even and odd columns in the two halves of a packed
// accumulator (packed fp32x2 instructions, explicit rounding), the halves
// added, then the xor butterfly; mean = sum / D, var = sum (x - mean)^2 / D,
// rstd = 1 / sqrt(var + eps), each operation rounded once.
// --------------------------------------------------------------------------
constexpr int kF32FwdVPL = kF32MaxD / 128;  // 32 vectors per lane at most

template <int VPL>
__global__ void __launch_bounds__(256, VPL <= 24 ? 2 : 1)
f32_out_fwd_kernel(const float *__restrict__ x, const float *__restrict__ emb, float *__restrict__ out,
                   float *__restrict__ mean, float *__restrict__ rstd, int S, int D, float eps, int rows_per_cta) {
    extern __shared__ __align__(16) float tab_f32[];  // onep [D], shift [D]
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.y;
    const int V = D / 4;
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i < D; i += blockDim.x) {
        tab_f32[i] = __fadd_rn(1.0f, emb[(size_t)b * 2 * D + i]);
        tab_f32[D + i] = emb[(size_t)b * 2 * D + D + i];
    }
    __syncthreads();
    const float4 *po = reinterpret_cast<const float4 *>(tab_f32);
    const float4 *ps = reinterpret_cast<const float4 *>(tab_f32 + D);
    const float Df = (float)D;
    const int s_begin = blockIdx.x * rows_per_cta;
    const int s_end = min(S, s_begin + rows_per_cta);
    const uint64_t pol = l2_evict_first();
    for (int s = s_begin + warp; s < s_end; s += 8) {
        const size_t row = (size_t)b * S + s;
        const float *xr = x + row * D;
        float4 xv[VPL];
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int v = lane + 32 * j;
            xv[j] = v < V ? ldf4_hint(xr + (size_t)v * 4, pol) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        // sums by column pair (packed), the halves added, then the butterfly
        px2 s1 = 0ull;
#pragma unroll
        for (int j = 0; j < VPL; ++j)
            if (lane + 32 * j < V)
                s1 = px_add(px_add(s1, px_make(xv[j].x, xv[j].y)), px_make(xv[j].z, xv[j].w));
        const float mu = __fdiv_rn(warp_sum(__fadd_rn(px_lo(s1), px_hi(s1))), Df);
        const px2 mu2 = px_splat(mu);
        px2 s2 = 0ull;
#pragma unroll
        for (int j = 0; j < VPL; ++j)
            if (lane + 32 * j < V) {
                const px2 d0 = px_sub(px_make(xv[j].x, xv[j].y), mu2);
                const px2 d1 = px_sub(px_make(xv[j].z, xv[j].w), mu2);
                s2 = px_add(px_add(s2, px_mul(d0, d0)), px_mul(d1, d1));
            }
        const float var = __fdiv_rn(warp_sum(__fadd_rn(px_lo(s2), px_hi(s2))), Df);
        const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(var, eps)));
        const px2 rs2 = px_splat(rs);
        if (lane == 0) {
            mean[row] = mu;
            rstd[row] = rs;
        }
        float4 *orow = reinterpret_cast<float4 *>(out + row * D);
        // out = fp32(fp32(fp32(fp32(x - mean) * rstd) * onep) + shift)
        auto mod = [&](float a, float b, float on_a, float on_b, float sh_a, float sh_b) {
            return px_add(px_mul(px_mul(px_sub(px_make(a, b), mu2), rs2), px_make(on_a, on_b)), px_make(sh_a, sh_b));
        };
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int v = lane + 32 * j;
            if (v < V) {
                const float4 a = xv[j], on = po[v], sh = ps[v];
                const px2 lo = mod(a.x, a.y, on.x, on.y, sh.x, sh.y), hi = mod(a.z, a.w, on.z, on.w, sh.z, sh.w);
                stg16f_hint(orow + v, make_float4(px_lo(lo), px_hi(lo), px_lo(hi), px_hi(hi)), pol);
            }
        }
    }
}

// --------------------------------------------------------------------------
// LayerNorm + modulation backward and the level-0 tree tiles: one CTA per
// (sample b, 32-token tile t); thread i owns the float4 vectors i + NT j
// (j < VPT: three per thread up to D = 3072, four up to 4096).  Per row in ascending s: xhat = fp32(fp32(x - mean) * rstd), g = dy,
// p = fp32(g * xhat) and g go into the columns' tiles by TwoSum from (+0, +0);
// each thread's fused multiply-add sums of g * onep and p * onep over its
// columns (even and odd columns in the two halves of a packed accumulator,
// then added), the warp butterfly, the warps in ascending order: c1, c2
// (divided by D); dx = fp32(rstd * fp32(fp32(gh - c1) - fp32(xhat * c2))).
// All arithmetic on column pairs in packed fp32x2 instructions with explicit
// rounding (a float4 of a row is two pairs as loaded).  Two CTAs per SM hide
// the loads' latency.
// --------------------------------------------------------------------------
// EXACT: D / 4 == blockDim.x * VPT, every thread's vectors inside the row (no tests)
template <int VPT, int MAXNT, bool EXACT>
__global__ void __launch_bounds__(MAXNT, 2)
f32_out_bwd_tile_kernel(const float *__restrict__ dy, const float *__restrict__ x, const float *__restrict__ emb,
                        const float *__restrict__ mean, const float *__restrict__ rstd, float *__restrict__ dx,
                        float *__restrict__ ws_sig, float *__restrict__ ws_kap, int S, int D, int T) {
    __shared__ float2 red[2][32];
    const int tid = threadIdx.x;
    const int NT = blockDim.x;
    const int nw = NT >> 5;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int t = blockIdx.x;
    const int b = blockIdx.y;
    const int V = D / 4;
    const int H = 2 * D;
    pdl_wait();
    pdl_trigger();
    // onep = fp32(1 + scale) of this thread's columns, by column pair
    px2 onep[VPT][2];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tid + NT * j;
        float4 sc = make_float4(-1.0f, -1.0f, -1.0f, -1.0f);
        if (EXACT || v < V) sc = reinterpret_cast<const float4 *>(emb + (size_t)b * 2 * D)[v];
        onep[j][0] = px_make(__fadd_rn(1.0f, sc.x), __fadd_rn(1.0f, sc.y));
        onep[j][1] = px_make(__fadd_rn(1.0f, sc.z), __fadd_rn(1.0f, sc.w));
    }
    // tree nodes of the scale products p and of the shift products g, by
    // column pair, from (+0, +0)
    px2 ss[VPT][2], ks[VPT][2], sh[VPT][2], kh[VPT][2];
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int c = 0; c < 2; ++c) ss[j][c] = ks[j][c] = sh[j][c] = kh[j][c] = 0ull;
    const int s0 = t * kTile;
    const int n = min(kTile, S - s0);
    const float Df = (float)D;
    const uint64_t pol = l2_evict_first();
    for (int i = 0; i < n; ++i) {
        const size_t row = (size_t)b * S + s0 + i;
        px2 xp[VPT][2], gp[VPT][2];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = tid + NT * j;
            uint4 xw = make_uint4(0u, 0u, 0u, 0u), gw = xw;
            if (EXACT || v < V) {
                xw = ldg16_hint(x + row * D + (size_t)v * 4, pol);
                gw = ldg16_hint(dy + row * D + (size_t)v * 4, pol);
            }
            xp[j][0] = px_make(__uint_as_float(xw.x), __uint_as_float(xw.y));
            xp[j][1] = px_make(__uint_as_float(xw.z), __uint_as_float(xw.w));
            gp[j][0] = px_make(__uint_as_float(gw.x), __uint_as_float(gw.y));
            gp[j][1] = px_make(__uint_as_float(gw.z), __uint_as_float(gw.w));
        }
        const float mu = mean[row], rs = rstd[row];
        const px2 mu2 = px_splat(mu), rs2 = px_splat(rs);
        // phase 1: x_hat, the tree products and this thread's row sums (column
        // pairs in packed fused multiply-adds, the halves added at the end)
        px2 a1 = 0ull, a2 = 0ull;
        px2 xh[VPT][2];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            if (EXACT || tid + NT * j < V) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    xh[j][c] = px_mul(px_sub(xp[j][c], mu2), rs2);
                    const px2 p = px_mul(gp[j][c], xh[j][c]);
                    px_twosum(ss[j][c], ks[j][c], p);
                    px_twosum(sh[j][c], kh[j][c], gp[j][c]);
                    a1 = px_fma(gp[j][c], onep[j][c], a1);
                    a2 = px_fma(p, onep[j][c], a2);
                }
            } else {
                xh[j][0] = xh[j][1] = 0ull;
            }
        }
        const float s1 = warp_sum(__fadd_rn(px_lo(a1), px_hi(a1)));
        const float s2 = warp_sum(__fadd_rn(px_lo(a2), px_hi(a2)));
        if (lane == 0) red[i & 1][warp] = make_float2(s1, s2);
        __syncthreads();
        float t1 = red[i & 1][0].x, t2 = red[i & 1][0].y;
        for (int w = 1; w < nw; ++w) t1 = __fadd_rn(t1, red[i & 1][w].x), t2 = __fadd_rn(t2, red[i & 1][w].y);
        const px2 c1 = px_splat(__fdiv_rn(t1, Df)), c2 = px_splat(__fdiv_rn(t2, Df));
        // phase 2: dx = fp32(rstd * fp32(fp32(gh - c1) - fp32(x_hat * c2))), gh = fp32(g * onep)
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = tid + NT * j;
            if (EXACT || v < V) {
                px2 o[2];
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const px2 gh = px_mul(gp[j][c], onep[j][c]);
                    o[c] = px_mul(rs2, px_sub(px_sub(gh, c1), px_mul(xh[j][c], c2)));
                }
                stg16f_hint(dx + row * D + (size_t)v * 4, make_float4(px_lo(o[0]), px_hi(o[0]), px_lo(o[1]), px_hi(o[1])),
                            pol);
            }
        }
        // red[i & 1] is written again two rows later, after the next barrier
    }
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tid + NT * j;
        if (EXACT || v < V) {
            const size_t node = ((size_t)b * T + t) * H + (size_t)v * 4;
            stg16f(ws_sig + node, make_float4(px_lo(ss[j][0]), px_hi(ss[j][0]), px_lo(ss[j][1]), px_hi(ss[j][1])));
            stg16f(ws_kap + node, make_float4(px_lo(ks[j][0]), px_hi(ks[j][0]), px_lo(ks[j][1]), px_hi(ks[j][1])));
            stg16f(ws_sig + node + D, make_float4(px_lo(sh[j][0]), px_hi(sh[j][0]), px_lo(sh[j][1]), px_hi(sh[j][1])));
            stg16f(ws_kap + node + D, make_float4(px_lo(kh[j][0]), px_hi(kh[j][0]), px_lo(kh[j][1]), px_hi(kh[j][1])));
        }
    }
}

// --------------------------------------------------------------------------
// Projection backward: one CTA per (256 columns, 256-row slab of W).  A thread
// owns 4 consecutive columns (one float4 of every row) and one of 4 row groups
// of the slab (rows rg, rg + 4, ...).  Over its rows ascending: d_silu partials
// ds[b] = fma(e[b,n], W[n,k], ds[b]); the slab's partial is the four groups'
// added in ascending group order (written per slab: ws[slab][b][k]).  The
// weight gradient acc = fma(e[b,n], u[b,k], acc) over the samples ascending,
// starting from the accumulator (accumulate) or +0; db likewise with
// additions.  Samples in chunks of kF32BC; a later chunk continues from the
// accumulator the earlier one wrote.  All orders depend on D only.
// --------------------------------------------------------------------------
constexpr int kF32Slab = 256;
constexpr int kF32RowGroups = 4;
constexpr int kF32SlabRowsInFlight = 8;  // rows of W (a float4 each) each thread has requested at once

__device__ __forceinline__ float4 ldf4(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}
__device__ __forceinline__ float4 fma4(float a, float4 b, float4 c) {
    return make_float4(__fmaf_rn(a, b.x, c.x), __fmaf_rn(a, b.y, c.y), __fmaf_rn(a, b.z, c.z),
                       __fmaf_rn(a, b.w, c.w));
}
__device__ __forceinline__ float4 add4(float4 a, float4 b) {
    return make_float4(__fadd_rn(a.x, b.x), __fadd_rn(a.y, b.y), __fadd_rn(a.z, b.z), __fadd_rn(a.w, b.w));
}

__global__ void __launch_bounds__(256, 2)
f32_proj_bwd_slab_kernel(const float *__restrict__ d_emb, const float *__restrict__ u, const float *__restrict__ W,
                         float *__restrict__ dW_acc, float *__restrict__ db_acc, int accumulate,
                         float *__restrict__ ws, int B, int D) {
    __shared__ float es[kF32BC][kF32Slab];
    __shared__ float4 part[kF32RowGroups - 1][kF32BC][64];  // row groups 1..3's partials
    const int ct = threadIdx.x & 63;
    const int rg = threadIdx.x >> 6;
    const int k = blockIdx.x * 256 + ct * 4;  // the first of this thread's 4 columns
    const int slab = blockIdx.y;
    const int N = 2 * D;
    const int n0 = slab * kF32Slab;
    const int rows = min(kF32Slab, N - n0);
    const int nrow = rows > rg ? (rows - rg + kF32RowGroups - 1) / kF32RowGroups : 0;  // rows of this group
    const bool live = k < D;  // D % 4 == 0: all 4 columns inside D
    pdl_wait();
    pdl_trigger();
    for (int b0 = 0; b0 < B; b0 += kF32BC) {
        const int nb = min(kF32BC, B - b0);
        __syncthreads();
        for (int i = threadIdx.x; i < kF32BC * kF32Slab; i += blockDim.x) {
            const int bb = i / kF32Slab, r = i % kF32Slab;
            es[bb][r] = (bb < nb && r < rows) ? d_emb[(size_t)(b0 + bb) * N + n0 + r] : 0.0f;
        }
        __syncthreads();
        float4 uk[kF32BC], ds[kF32BC];
#pragma unroll
        for (int bb = 0; bb < kF32BC; ++bb) {
            uk[bb] = (live && bb < nb) ? ldf4(u + (size_t)(b0 + bb) * D + k) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            ds[bb] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
        const bool first = b0 == 0 && !accumulate;
        const float *wcol = W + (size_t)(n0 + rg) * D + k;
        float *acol = dW_acc ? dW_acc + (size_t)(n0 + rg) * D + k : nullptr;
        const size_t step = (size_t)kF32RowGroups * D;  // from one row of the group to the next
        for (int i0 = 0; i0 < nrow; i0 += kF32SlabRowsInFlight) {
            float4 w[kF32SlabRowsInFlight];  // requested before the first use
#pragma unroll
            for (int q = 0; q < kF32SlabRowsInFlight; ++q)
                w[q] = (live && i0 + q < nrow) ? ldf4(wcol + (size_t)(i0 + q) * step)
                                               : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
            for (int q = 0; q < kF32SlabRowsInFlight; ++q) {
                const int i = i0 + q;
                if (i < nrow) {
                    const int r = rg + kF32RowGroups * i;
#pragma unroll
                    for (int bb = 0; bb < kF32BC; ++bb)
                        if (bb < nb) ds[bb] = fma4(es[bb][r], w[q], ds[bb]);
                    if (acol && live) {
                        float4 *pa = reinterpret_cast<float4 *>(acol + (size_t)i * step);
                        float4 a = first ? make_float4(0.0f, 0.0f, 0.0f, 0.0f) : *pa;
#pragma unroll
                        for (int bb = 0; bb < kF32BC; ++bb)
                            if (bb < nb) a = fma4(es[bb][r], uk[bb], a);
                        *pa = a;
                    }
                }
            }
        }
        // the slab's partial: row groups added in ascending order
        if (rg > 0)
#pragma unroll
            for (int bb = 0; bb < kF32BC; ++bb) part[rg - 1][bb][ct] = ds[bb];
        __syncthreads();
        if (rg == 0 && live)
#pragma unroll
            for (int bb = 0; bb < kF32BC; ++bb)
                if (bb < nb) {
                    float4 t = ds[bb];
#pragma unroll
                    for (int g = 1; g < kF32RowGroups; ++g) t = add4(t, part[g - 1][bb][ct]);
                    __stcg(reinterpret_cast<float4 *>(ws + ((size_t)slab * B + b0 + bb) * D + k), t);
                }
        if (db_acc && blockIdx.x == 0)
            for (int r = threadIdx.x; r < rows; r += blockDim.x) {
                float a = first ? 0.0f : db_acc[n0 + r];
                for (int bb = 0; bb < nb; ++bb) a = __fadd_rn(a, es[bb][r]);
                db_acc[n0 + r] = a;
            }
    }
}

// d_temb[b,k] = fp32((sum over slabs, ascending) * silu'(t)), the product in fp64
__global__ void __launch_bounds__(256)
f32_proj_bwd_final_kernel(const float *__restrict__ ws, const float *__restrict__ temb, float *__restrict__ d_temb,
                          int B, int D, int nslab) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long BD = (long long)B * D;
    // silu'(t) in fp64 before the wait (temb is an input of this call; the
    // kernel before this one is the call's own slab kernel, which cannot write
    // it, and which started only after all earlier work had completed)
    double dsl = 0.0;
    if (i < BD) {
        const double x = (double)temb[i];
        const double sg = 1.0 / (1.0 + exp(-x));
        dsl = sg * (1.0 + x * (1.0 - sg));
    }
    pdl_wait();
    pdl_trigger();
    if (i < BD) {
        constexpr int kMax = 2 * kF32MaxD / kF32Slab;  // 32 slabs at most
        float part[kMax];
#pragma unroll
        for (int s = 0; s < kMax; ++s) part[s] = s < nslab ? __ldcg(ws + (size_t)s * BD + i) : 0.0f;
        float tot = part[0];
#pragma unroll
        for (int s = 1; s < kMax; ++s)
            if (s < nslab) tot = __fadd_rn(tot, part[s]);
        d_temb[i] = (float)((double)tot * dsl);
    }
}

// --------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------
cudaError_t launch_f32_proj_fwd(const float *temb, const float *W, const float *bias, float *emb, float *u, int B,
                                int D, cudaStream_t stream, const DeviceInfo &dev) {
    const long long n = (long long)B * D;
    cudaError_t err = launch_pdl(f32_silu_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, stream, temb, u, n);
    if (err != cudaSuccess) return err;
    const size_t smem = (size_t)kF32BC * D * 4;
    err = ensure_smem_attr((const void *)f32_proj_fwd_kernel, smem, dev);
    if (err != cudaSuccess) return err;
    return launch_pdl(f32_proj_fwd_kernel, dim3((unsigned)((2 * D + 7) / 8)), dim3(256), smem, stream, u, W, bias,
                      emb, B, D);
}

cudaError_t launch_f32_out_fwd(const float *x, const float *emb, float *out, float *mean, float *rstd, int B, int S,
                               int D, float eps, cudaStream_t stream, const DeviceInfo &dev) {
    const size_t smem = (size_t)2 * D * 4;
    // about four CTAs of 8 warps per SM over the batch
    int cps = (dev.sm_count * 4 + B - 1) / B;
    if (cps > (S + 7) / 8) cps = (S + 7) / 8;
    if (cps < 1) cps = 1;
    const int rows = (S + cps - 1) / cps;
    const dim3 grid((unsigned)((S + rows - 1) / rows), (unsigned)B);
    if (D / 4 <= 32 * 24) {  // D <= 3072: 24 vectors per lane, two CTAs per SM
        cudaError_t err = ensure_smem_attr((const void *)f32_out_fwd_kernel<24>, smem, dev);
        if (err != cudaSuccess) return err;
        return launch_pdl(f32_out_fwd_kernel<24>, grid, dim3(256), smem, stream, x, emb, out, mean, rstd, S, D, eps,
                          rows);
    }
    auto kern = f32_out_fwd_kernel<kF32FwdVPL>;
    cudaError_t err = ensure_smem_attr((const void *)kern, smem, dev);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, grid, dim3(256), smem, stream, x, emb, out, mean, rstd, S, D, eps, rows);
}

cudaError_t launch_f32_out_bwd(const float *dy, const float *x, const float *emb, const float *mean,
                               const float *rstd, float *dx, float *d_emb, void *ws, int B, int S, int D,
                               cudaStream_t stream, const DeviceInfo &dev) {
    if (S == 0) return launch_zero(d_emb, (size_t)B * 2 * D, stream);
    const int T = (S + kTile - 1) / kTile;
    const int H = 2 * D;
    float *sig = static_cast<float *>(ws);
    float *kap = sig + (size_t)B * T * H;
    // two CTAs per SM: three vectors (12 columns: more independent TwoSum
    // chains per thread) per thread up to D = 3072 (at most 256 threads), four
    // up to D = 4096 (at most 256)
    const int V = D / 4;
    cudaError_t err;
    if (V <= 768) {
        const int nt = ((V + 2) / 3 + 31) / 32 * 32;
        auto kern = nt * 3 == V ? f32_out_bwd_tile_kernel<3, 256, true> : f32_out_bwd_tile_kernel<3, 256, false>;
        err = launch_pdl(kern, dim3((unsigned)T, (unsigned)B), dim3(nt), 0, stream, dy, x, emb, mean, rstd, dx, sig,
                         kap, S, D, T);
    } else {
        const int nt = ((V + 3) / 4 + 31) / 32 * 32;
        auto kern = f32_out_bwd_tile_kernel<4, 256, false>;  // the exact form spills at 128 registers
        err = launch_pdl(kern, dim3((unsigned)T, (unsigned)B), dim3(nt), 0, stream, dy, x, emb, mean, rstd, dx, sig,
                         kap, S, D, T);
    }
    if (err != cudaSuccess) return err;
    return launch_fold(sig, kap, d_emb, B, T, H, stream, dev);
}

size_t f32_proj_bwd_ws_bytes(int B, int D) {
    const size_t nslab = (size_t)(2 * D + kF32Slab - 1) / kF32Slab;
    return nslab * (size_t)B * D * 4;
}

cudaError_t launch_f32_proj_bwd(const float *d_emb, const float *temb, const float *u, const float *W,
                                float *d_temb, float *dW_acc, float *db_acc, int accumulate, void *ws, int B, int D,
                                cudaStream_t stream, const DeviceInfo &dev) {
    (void)dev;
    const int nslab = (2 * D + kF32Slab - 1) / kF32Slab;
    float *part = static_cast<float *>(ws);
    cudaError_t err = launch_pdl(f32_proj_bwd_slab_kernel, dim3((unsigned)((D + 255) / 256), (unsigned)nslab),
                                 dim3(256), 0, stream, d_emb, u, W, dW_acc, db_acc, accumulate, part, B, D);
    if (err != cudaSuccess) return err;
    const long long BD = (long long)B * D;
    return launch_pdl(f32_proj_bwd_final_kernel, dim3((unsigned)((BD + 255) / 256)), dim3(256), 0, stream, part, temb,
                      d_temb, B, D, nslab);
}

}  // namespace adaln

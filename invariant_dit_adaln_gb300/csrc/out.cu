// LayerNorm + modulation forward, fused LayerNorm backward with the level-0
// token-tree tiles, the tree fold, and the standalone token tree.
//
// Operator: RL-Kernel PR 538 "final_adaln_out", section "What"; rounding points:
// miles_diffusion PR 108, Summary, root cause 1; token tree: PR 538 "What" and
// the review thread on the cancellation case (Neumaier 32-token tiles, folded
// level by level, one final add).
//
// Layout in HBM (all dense, row-major):
//   x, dy, out, dx   [B, S, D] bf16     one token row = D * 2 bytes, 16-B aligned
//   emb              [B, 2D]   bf16     [scale | shift]
//   mean, rstd       [B, S]    fp32
//   d_emb            [B, 2D]   fp32     [d_scale | d_shift]
//   tree partials    sigma [B, T, H] fp32 then kappa [B, T, H] fp32, T = ceil(S/32)
#include "common.cuh"
#include "internal.h"

namespace adaln {

static __device__ unsigned g_err;  // device-side error word (see adaln_device_error)

__device__ __forceinline__ void report_error(unsigned code) { atomicCAS(&g_err, 0u, code); }

// ==========================================================================
// Forward: one warp-group (128 threads) per token row, persistent.
//
// A CTA holds kWG warp-groups; each owns a contiguous range of rows and a ring
// of K row buffers in shared memory, filled by 1-D bulk copies (the TMA
// engine) that one thread issues K rows ahead.  Thread t of a warp-group owns
// the 16-byte vectors v = t + 128 j (8 columns each) of every row, so its
// modulation parameters stay in registers while the sample index is unchanged.
// The reduction order over d: per thread in (j, element) order, a fixed xor
// butterfly within the warp, then the four warps in ascending order.  It
// depends on D only.
// ==========================================================================
constexpr int kWG = 2;            // warp-groups per CTA
constexpr int kFwdStages = 4;     // rows in flight per warp-group

template <int VPT>
struct FwdSmem {
    // per warp-group: [slot 0/1][sum, sq][warp 0..3]
    float red[kWG][2][2][4];
    uint64_t full[kWG][kFwdStages];
};

template <int VPT>
__global__ void __launch_bounds__(kWG * 128)
out_fwd_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ emb, uint16_t *__restrict__ out,
               float *__restrict__ mean, float *__restrict__ rstd, int S, int D, float eps, long long R) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    FwdSmem<VPT> &sm = *reinterpret_cast<FwdSmem<VPT> *>(smem_raw);
    const int row_bytes = D * 2;
    unsigned char *stages = smem_raw + ((sizeof(FwdSmem<VPT>) + 127) / 128) * 128;

    const int wg = threadIdx.x >> 7;
    const int t = threadIdx.x & 127;
    const int warp = t >> 5;
    const int lane = t & 31;
    const int V = D >> 3;
    unsigned char *my_stages = stages + (size_t)wg * kFwdStages * row_bytes;

    const long long G = (long long)gridDim.x * kWG;
    const long long g = (long long)blockIdx.x * kWG + wg;
    const long long r_begin = (g * R) / G;
    const long long r_end = ((g + 1) * R) / G;
    const int nrows = (int)(r_end - r_begin);

    if (t == 0) {
        for (int s = 0; s < kFwdStages; ++s) mbar_init(&sm.full[wg][s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();  // inputs may come from the preceding kernel

    if (t == 0) {
        for (int i = 0; i < kFwdStages && i < nrows; ++i) {
            mbar_arrive_expect_tx(&sm.full[wg][i], row_bytes);
            bulk_g2s(my_stages + (size_t)i * row_bytes, x + (size_t)(r_begin + i) * D, row_bytes, &sm.full[wg][i]);
        }
    }

    uint32_t onep[VPT][4], shift[VPT][4];  // packed bf16x2 parameters of the current sample
    long long cur_b = -1;
    const float invD_num = (float)D;

    for (int i = 0; i < nrows; ++i) {
        const long long r = r_begin + i;
        const long long b = r / S;
        if (b != cur_b) {
            cur_b = b;
            const uint16_t *e = emb + (size_t)b * 2 * D;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = t + 128 * j;
                if (v < V) {
                    uint4 sc = ldg16(e + (size_t)v * 8);
                    uint4 sh = ldg16(e + D + (size_t)v * 8);
                    float f[8];
                    unpack8(sc, f);
                    float o[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) o[k] = __fadd_rn(1.0f, f[k]);
                    uint4 op = pack8(o);  // onep = bf16(fp32(1 + scale))
                    onep[j][0] = op.x; onep[j][1] = op.y; onep[j][2] = op.z; onep[j][3] = op.w;
                    shift[j][0] = sh.x; shift[j][1] = sh.y; shift[j][2] = sh.z; shift[j][3] = sh.w;
                }
            }
        }
        const int st = i % kFwdStages;
        const uint32_t parity = (uint32_t)(i / kFwdStages) & 1u;
        const bool ok = mbar_wait_bounded(&sm.full[wg][st], parity);

        float xv[VPT][8];
        float s1 = 0.0f;
        const unsigned char *row = my_stages + (size_t)st * row_bytes;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = t + 128 * j;
            if (v < V && ok) {
                uint4 w = *reinterpret_cast<const uint4 *>(row + (size_t)v * 16);
                unpack8(w, xv[j]);
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) xv[j][k] = 0.0f;
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) s1 = __fadd_rn(s1, xv[j][k]);
        }
        s1 = warp_sum(s1);
        const int slot = i & 1;
        if (lane == 0) sm.red[wg][slot][0][warp] = s1;
        // barrier of the warp-group, and a vote: did any thread time out?
        int bad;
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t"
            "setp.ne.u32 p, %1, 0;\n\t"
            "bar.red.or.pred q, %2, 128, p;\n\t"
            "selp.u32 %0, 1, 0, q;\n\t}"
            : "=r"(bad)
            : "r"((unsigned)!ok), "r"(1 + wg)
            : "memory");
        if (bad) {
            if (t == 0) {
                report_error(kErrOutFwdWait);
                // let the copies this warp-group issued finish before leaving
                const int issued = min(nrows, i + kFwdStages);
                for (int k = i; k < issued; ++k)
                    mbar_wait_bounded(&sm.full[wg][k % kFwdStages], (uint32_t)(k / kFwdStages) & 1u, 10000000ull);
            }
            return;
        }
        // every thread of the warp-group has read stage st: refill it
        if (t == 0 && i + kFwdStages < nrows) {
            mbar_arrive_expect_tx(&sm.full[wg][st], row_bytes);
            bulk_g2s(my_stages + (size_t)st * row_bytes, x + (size_t)(r + kFwdStages) * D, row_bytes,
                     &sm.full[wg][st]);
        }
        float tot = sm.red[wg][slot][0][0];
        tot = __fadd_rn(tot, sm.red[wg][slot][0][1]);
        tot = __fadd_rn(tot, sm.red[wg][slot][0][2]);
        tot = __fadd_rn(tot, sm.red[wg][slot][0][3]);
        const float mu = __fdiv_rn(tot, invD_num);

        float s2 = 0.0f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = t + 128 * j;
            if (v < V) {
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float c = __fsub_rn(xv[j][k], mu);
                    s2 = __fadd_rn(s2, __fmul_rn(c, c));
                }
            }
        }
        s2 = warp_sum(s2);
        if (lane == 0) sm.red[wg][slot][1][warp] = s2;
        named_bar(1 + wg, 128);
        float tq = sm.red[wg][slot][1][0];
        tq = __fadd_rn(tq, sm.red[wg][slot][1][1]);
        tq = __fadd_rn(tq, sm.red[wg][slot][1][2]);
        tq = __fadd_rn(tq, sm.red[wg][slot][1][3]);
        const float var = __fdiv_rn(tq, invD_num);
        const float rs = __frsqrt_rn(__fadd_rn(var, eps));

        uint16_t *orow = out + (size_t)r * D;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = t + 128 * j;
            if (v < V) {
                float o[8];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float xh0 = __fmul_rn(__fsub_rn(xv[j][2 * q], mu), rs);
                    const float xh1 = __fmul_rn(__fsub_rn(xv[j][2 * q + 1], mu), rs);
                    o[2 * q] = __fadd_rn(__fmul_rn(xh0, bf16lo(onep[j][q])), bf16lo(shift[j][q]));
                    o[2 * q + 1] = __fadd_rn(__fmul_rn(xh1, bf16hi(onep[j][q])), bf16hi(shift[j][q]));
                }
                stg16(orow + (size_t)v * 8, pack8(o));
            }
        }
        if (t == 0) {
            mean[r] = mu;
            rstd[r] = rs;
        }
    }
    pdl_trigger();
}

template <int VPT>
static cudaError_t launch_out_fwd_t(const uint16_t *x, const uint16_t *emb, uint16_t *out, float *mean,
                                    float *rstd, int B, int S, int D, float eps, cudaStream_t stream,
                                    const DeviceInfo &dev) {
    const size_t smem = ((sizeof(FwdSmem<VPT>) + 127) / 128) * 128 + (size_t)kWG * kFwdStages * D * 2;
    auto kern = out_fwd_kernel<VPT>;
    cudaError_t err = ensure_smem_attr((const void *)kern, smem, dev);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWG * 128, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    const long long R = (long long)B * S;
    long long grid = (long long)dev.sm_count * per_sm;
    const long long need = (R + kWG - 1) / kWG;
    if (grid > need) grid = need;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kWG * 128), smem, stream,
                      x, emb, out, mean, rstd, S, D, eps, R);
}

cudaError_t launch_out_fwd(const uint16_t *x, const uint16_t *emb, uint16_t *out, float *mean, float *rstd,
                           int B, int S, int D, float eps, cudaStream_t stream, const DeviceInfo &dev) {
    const int V = D / 8;
    const int vpt = (V + 127) / 128;
    switch (vpt) {
        case 1: return launch_out_fwd_t<1>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev);
        case 2: return launch_out_fwd_t<2>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev);
        case 3: return launch_out_fwd_t<3>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev);
        case 4: return launch_out_fwd_t<4>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev);
        case 5: case 6: return launch_out_fwd_t<6>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev);
        default: return launch_out_fwd_t<8>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev);
    }
}

// ==========================================================================
// Backward, kernel 1: one CTA per (sample b, 32-token tile t).
//
// Thread i owns the 16-byte vectors v = i + NT j (8 columns each).  The CTA
// walks the tile's rows in ascending s.  Per row it forms gh = g * onep and
// xhat (bit-identical to the forward's), reduces sum(gh) and sum(gh * xhat)
// over the row (per thread in (j, element) order, a fixed butterfly, then the
// warps in ascending order), writes dx, and adds the products g * xhat and g
// into per-column Neumaier accumulators: the tile's level-0 node of the tree.
// Rows arrive through a ring of bulk copies (x row and dy row per stage).
// ==========================================================================
constexpr int kBwdStages = 4;

struct BwdSmem {
    float red[2][2][32];      // [slot][sum gh, sum gh*xhat][warp]
    float mu[kTile], rs[kTile];
    uint64_t full[kBwdStages];
};

template <int VPT, int MAXNT, int MINB>
__global__ void __launch_bounds__(MAXNT, MINB)
out_bwd_tile_kernel(const uint16_t *__restrict__ dy, const uint16_t *__restrict__ x,
                    const uint16_t *__restrict__ emb, const float *__restrict__ mean,
                    const float *__restrict__ rstd, uint16_t *__restrict__ dx, float *__restrict__ ws_sig,
                    float *__restrict__ ws_kap, int S, int D, int T) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    BwdSmem &sm = *reinterpret_cast<BwdSmem *>(smem_raw);
    unsigned char *stages = smem_raw + ((sizeof(BwdSmem) + 127) / 128) * 128;
    const int row_bytes = D * 2;
    const int stage_bytes = 2 * row_bytes;  // x row, then dy row

    const int tile = blockIdx.x;
    const int b = blockIdx.y;
    const int NT = blockDim.x;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int nwarps = NT >> 5;
    const int V = D >> 3;
    const int s0 = tile * kTile;
    const int n = min(kTile, S - s0);
    const size_t row0 = (size_t)b * S + s0;

    if (tid == 0) {
        for (int s = 0; s < kBwdStages; ++s) mbar_init(&sm.full[s], 1);
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();

    if (tid == 0) {
        for (int i = 0; i < kBwdStages && i < n; ++i) {
            unsigned char *dst = stages + (size_t)i * stage_bytes;
            mbar_arrive_expect_tx(&sm.full[i], stage_bytes);
            bulk_g2s(dst, x + (row0 + i) * D, row_bytes, &sm.full[i]);
            bulk_g2s(dst + row_bytes, dy + (row0 + i) * D, row_bytes, &sm.full[i]);
        }
    }
    if (tid < n) {
        sm.mu[tid] = mean[row0 + tid];
        sm.rs[tid] = rstd[row0 + tid];
    }
    float onep[VPT][8];
    const uint16_t *e = emb + (size_t)b * 2 * D;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tid + NT * j;
        if (v < V) {
            uint4 sc = ldg16(e + (size_t)v * 8);
            float f[8];
            unpack8(sc, f);
#pragma unroll
            for (int k = 0; k < 8; ++k) onep[j][k] = bf16f(bf16_bits(__fadd_rn(1.0f, f[k])));
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) onep[j][k] = 0.0f;
        }
    }
    __syncthreads();

    float sg_s[VPT][8], kp_s[VPT][8];  // tree node for the scale products g * xhat
    float sg_h[VPT][8], kp_h[VPT][8];  // tree node for the shift products g
    const float Df = (float)D;

    for (int i = 0; i < n; ++i) {
        const int st = i % kBwdStages;
        const bool ok = mbar_wait_bounded(&sm.full[st], (uint32_t)(i / kBwdStages) & 1u);
        const unsigned char *xs = stages + (size_t)st * stage_bytes;
        const unsigned char *gs = xs + row_bytes;
        const float mu = sm.mu[i], rs = sm.rs[i];

        float xh[VPT][8], g[VPT][8];
        float a1 = 0.0f, a2 = 0.0f;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = tid + NT * j;
            if (v < V && ok) {
                float xf[8];
                unpack8(*reinterpret_cast<const uint4 *>(xs + (size_t)v * 16), xf);
                unpack8(*reinterpret_cast<const uint4 *>(gs + (size_t)v * 16), g[j]);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    xh[j][k] = __fmul_rn(__fsub_rn(xf[k], mu), rs);
                    const float gh = __fmul_rn(g[j][k], onep[j][k]);
                    a1 = __fadd_rn(a1, gh);
                    a2 = __fadd_rn(a2, __fmul_rn(gh, xh[j][k]));
                }
            } else {
#pragma unroll
                for (int k = 0; k < 8; ++k) { xh[j][k] = 0.0f; g[j][k] = 0.0f; }
            }
        }
        a1 = warp_sum(a1);
        a2 = warp_sum(a2);
        const int slot = i & 1;
        if (lane == 0) {
            sm.red[slot][0][warp] = a1;
            sm.red[slot][1][warp] = a2;
        }
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                report_error(kErrOutBwdWait);
                const int issued = min(n, i + kBwdStages);
                for (int k = i; k < issued; ++k)
                    mbar_wait_bounded(&sm.full[k % kBwdStages], (uint32_t)(k / kBwdStages) & 1u, 10000000ull);
            }
            return;
        }
        if (tid == 0 && i + kBwdStages < n) {
            unsigned char *dst = stages + (size_t)st * stage_bytes;
            mbar_arrive_expect_tx(&sm.full[st], stage_bytes);
            bulk_g2s(dst, x + (row0 + i + kBwdStages) * D, row_bytes, &sm.full[st]);
            bulk_g2s(dst + row_bytes, dy + (row0 + i + kBwdStages) * D, row_bytes, &sm.full[st]);
        }
        float c1 = sm.red[slot][0][0], c2 = sm.red[slot][1][0];
        for (int w = 1; w < nwarps; ++w) {
            c1 = __fadd_rn(c1, sm.red[slot][0][w]);
            c2 = __fadd_rn(c2, sm.red[slot][1][w]);
        }
        c1 = __fdiv_rn(c1, Df);
        c2 = __fdiv_rn(c2, Df);

        uint16_t *drow = dx + (row0 + i) * D;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = tid + NT * j;
            if (v < V) {
                float o[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float gh = __fmul_rn(g[j][k], onep[j][k]);
                    o[k] = __fmul_rn(rs, __fsub_rn(__fsub_rn(gh, c1), __fmul_rn(xh[j][k], c2)));
                    const float ps = __fmul_rn(g[j][k], xh[j][k]);
                    if (i == 0) {
                        sg_s[j][k] = ps; kp_s[j][k] = 0.0f;
                        sg_h[j][k] = g[j][k]; kp_h[j][k] = 0.0f;
                    } else {
                        neumaier(sg_s[j][k], kp_s[j][k], ps);
                        neumaier(sg_h[j][k], kp_h[j][k], g[j][k]);
                    }
                }
                stg16(drow + (size_t)v * 8, pack8(o));
            }
        }
    }
    pdl_trigger();
    // level-0 node of this tile
    const int H = 2 * D;
    float *ps = ws_sig + ((size_t)b * T + tile) * H;
    float *pk = ws_kap + ((size_t)b * T + tile) * H;
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tid + NT * j;
        if (v < V) {
            const size_t c = (size_t)v * 8;
            stg16f(ps + c, make_float4(sg_s[j][0], sg_s[j][1], sg_s[j][2], sg_s[j][3]));
            stg16f(ps + c + 4, make_float4(sg_s[j][4], sg_s[j][5], sg_s[j][6], sg_s[j][7]));
            stg16f(pk + c, make_float4(kp_s[j][0], kp_s[j][1], kp_s[j][2], kp_s[j][3]));
            stg16f(pk + c + 4, make_float4(kp_s[j][4], kp_s[j][5], kp_s[j][6], kp_s[j][7]));
            stg16f(ps + D + c, make_float4(sg_h[j][0], sg_h[j][1], sg_h[j][2], sg_h[j][3]));
            stg16f(ps + D + c + 4, make_float4(sg_h[j][4], sg_h[j][5], sg_h[j][6], sg_h[j][7]));
            stg16f(pk + D + c, make_float4(kp_h[j][0], kp_h[j][1], kp_h[j][2], kp_h[j][3]));
            stg16f(pk + D + c + 4, make_float4(kp_h[j][4], kp_h[j][5], kp_h[j][6], kp_h[j][7]));
        }
    }
}

// ==========================================================================
// Standalone token tree, level 0: one thread per 4 columns of one tile.
// ==========================================================================
__global__ void __launch_bounds__(256)
tree_level0_kernel(const float *__restrict__ in, float *__restrict__ ws_sig, float *__restrict__ ws_kap,
                   int S, int H, int T) {
    pdl_wait();
    const int c4 = blockIdx.x * blockDim.x + threadIdx.x;
    const int tile = blockIdx.y;
    const int b = blockIdx.z;
    if (c4 * 4 >= H) return;
    const int s0 = tile * kTile;
    const int n = min(kTile, S - s0);
    const float *p = in + ((size_t)b * S + s0) * H + (size_t)c4 * 4;
    float s[4], c[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int i0 = 0; i0 < n; i0 += 8) {
        float4 v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (i0 + k < n) v[k] = __ldg(reinterpret_cast<const float4 *>(p + (size_t)(i0 + k) * H));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (i0 + k == 0) {
                s[0] = v[0].x; s[1] = v[0].y; s[2] = v[0].z; s[3] = v[0].w;
            } else if (i0 + k < n) {
                neumaier(s[0], c[0], v[k].x);
                neumaier(s[1], c[1], v[k].y);
                neumaier(s[2], c[2], v[k].z);
                neumaier(s[3], c[3], v[k].w);
            }
        }
    }
    pdl_trigger();
    const size_t o = ((size_t)b * T + tile) * H + (size_t)c4 * 4;
    stg16f(ws_sig + o, make_float4(s[0], s[1], s[2], s[3]));
    stg16f(ws_kap + o, make_float4(c[0], c[1], c[2], c[3]));
}

// ==========================================================================
// Tree fold: levels >= 1 and the final add.  One CTA per (sample, 32 columns);
// lane = column.  Warp w folds level-1 groups w, w + W, ... from the level-0
// partials in global memory; higher levels fold in shared memory.
// ==========================================================================
struct FoldSmem {
    float s1[kMaxLevel1][32], k1[kMaxLevel1][32];
    float s2[kMaxLevel1 / kTile][32], k2[kMaxLevel1 / kTile][32];
};

// one group of the fold: Neumaier sum of the children's sums in ascending
// order (compensation c), children's corrections added in ascending order;
// node = (sum, c + corrections)
__device__ __forceinline__ void fold_group(const float *sig, const float *kap, size_t stride, int count,
                                           float &out_s, float &out_k) {
    float s = 0.0f, c = 0.0f, k = 0.0f;
    for (int i0 = 0; i0 < count; i0 += 8) {
        float vs[8], vk[8];
#pragma unroll
        for (int q = 0; q < 8; ++q)
            if (i0 + q < count) {
                vs[q] = sig[(size_t)(i0 + q) * stride];
                vk[q] = kap[(size_t)(i0 + q) * stride];
            }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (i0 + q == 0) {
                s = vs[0];
                k = vk[0];
            } else if (i0 + q < count) {
                neumaier(s, c, vs[q]);
                k = __fadd_rn(k, vk[q]);
            }
        }
    }
    out_s = s;
    out_k = __fadd_rn(c, k);
}

__global__ void __launch_bounds__(1024)
tree_fold_kernel(const float *__restrict__ ws_sig, const float *__restrict__ ws_kap, float *__restrict__ out,
                 int T, int H) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    FoldSmem &sm = *reinterpret_cast<FoldSmem *>(smem_raw);
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    const int b = blockIdx.y;
    const int col = blockIdx.x * 32 + lane;
    const bool live = col < H;
    const size_t base = (size_t)b * T * H + (size_t)(live ? col : 0);

    if (T == 1) {  // the tile is the root
        if (warp == 0 && live) out[(size_t)b * H + col] = __fadd_rn(ws_sig[base], ws_kap[base]);
        pdl_trigger();
        return;
    }
    const int n1 = (T + kTile - 1) / kTile;
    for (int gi = warp; gi < n1; gi += W) {
        const int i0 = gi * kTile;
        const int cnt = min(kTile, T - i0);
        float s, k;
        fold_group(ws_sig + base + (size_t)i0 * H, ws_kap + base + (size_t)i0 * H, (size_t)H, cnt, s, k);
        sm.s1[gi][lane] = s;
        sm.k1[gi][lane] = k;
    }
    __syncthreads();
    // levels >= 2, alternating between the two shared buffers
    int nn = n1;
    bool in_first = true;
    while (nn > 1) {
        const int m = (nn + kTile - 1) / kTile;
        for (int gi = warp; gi < m; gi += W) {
            const int i0 = gi * kTile;
            const int cnt = min(kTile, nn - i0);
            float s, k;
            if (in_first) {
                fold_group(&sm.s1[i0][lane], &sm.k1[i0][lane], 32, cnt, s, k);
                sm.s2[gi][lane] = s;
                sm.k2[gi][lane] = k;
            } else {
                fold_group(&sm.s2[i0][lane], &sm.k2[i0][lane], 32, cnt, s, k);
                sm.s1[gi][lane] = s;
                sm.k1[gi][lane] = k;
            }
        }
        __syncthreads();
        in_first = !in_first;
        nn = m;
    }
    pdl_trigger();
    if (warp == 0 && live) {
        const float s = in_first ? sm.s1[0][lane] : sm.s2[0][lane];
        const float k = in_first ? sm.k1[0][lane] : sm.k2[0][lane];
        out[(size_t)b * H + col] = __fadd_rn(s, k);
    }
}

__global__ void zero_kernel(float *__restrict__ p, size_t n) {
    pdl_wait();
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) p[i] = 0.0f;
    pdl_trigger();
}

// --------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------
static cudaError_t launch_fold(const float *sig, const float *kap, float *out, int B, int T, int H,
                               cudaStream_t stream, const DeviceInfo &dev) {
    const int n1 = (T + kTile - 1) / kTile;
    const int warps = T == 1 ? 1 : min(32, n1);
    const size_t smem = sizeof(FoldSmem);
    cudaError_t err = ensure_smem_attr((const void *)tree_fold_kernel, smem, dev);
    if (err != cudaSuccess) return err;
    return launch_pdl(tree_fold_kernel, dim3((H + 31) / 32, B), dim3(32 * warps), smem, stream,
                      sig, kap, out, T, H);
}

static cudaError_t launch_zero(float *p, size_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    return launch_pdl(zero_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, stream, p, n);
}

template <int VPT, int MAXNT, int MINB>
static cudaError_t launch_out_bwd_t(const uint16_t *dy, const uint16_t *x, const uint16_t *emb, const float *mean,
                                    const float *rstd, uint16_t *dx, float *sig, float *kap, int B, int S, int D,
                                    int T, cudaStream_t stream, const DeviceInfo &dev) {
    const int V = D / 8;
    const int nt = ((V + VPT - 1) / VPT + 31) / 32 * 32;
    const size_t smem = ((sizeof(BwdSmem) + 127) / 128) * 128 + (size_t)kBwdStages * 4 * D;
    auto kern = out_bwd_tile_kernel<VPT, MAXNT, MINB>;
    cudaError_t err = ensure_smem_attr((const void *)kern, smem, dev);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(T, B), dim3(nt), smem, stream, dy, x, emb, mean, rstd, dx, sig, kap,
                      S, D, T);
}

cudaError_t launch_out_bwd(const uint16_t *dy, const uint16_t *x, const uint16_t *emb, const float *mean,
                           const float *rstd, uint16_t *dx, float *d_emb, void *ws, int B, int S, int D,
                           cudaStream_t stream, const DeviceInfo &dev) {
    if (S == 0) return launch_zero(d_emb, (size_t)B * 2 * D, stream);
    const int T = (S + kTile - 1) / kTile;
    const int H = 2 * D;
    float *sig = static_cast<float *>(ws);
    float *kap = sig + (size_t)B * T * H;
    const int V = D / 8;
    cudaError_t err;
    if (V <= 384)
        err = launch_out_bwd_t<1, 384, 2>(dy, x, emb, mean, rstd, dx, sig, kap, B, S, D, T, stream, dev);
    else if (V <= 512)
        err = launch_out_bwd_t<1, 512, 1>(dy, x, emb, mean, rstd, dx, sig, kap, B, S, D, T, stream, dev);
    else
        err = launch_out_bwd_t<2, 512, 1>(dy, x, emb, mean, rstd, dx, sig, kap, B, S, D, T, stream, dev);
    if (err != cudaSuccess) return err;
    return launch_fold(sig, kap, d_emb, B, T, H, stream, dev);
}

cudaError_t launch_token_tree(const float *in, float *out, void *ws, int B, int S, int H, cudaStream_t stream,
                              const DeviceInfo &dev) {
    if (S == 0) return launch_zero(out, (size_t)B * H, stream);
    const int T = (S + kTile - 1) / kTile;
    float *sig = static_cast<float *>(ws);
    float *kap = sig + (size_t)B * T * H;
    const int c4 = (H + 3) / 4;
    cudaError_t err = launch_pdl(tree_level0_kernel, dim3((c4 + 255) / 256, T, B), dim3(256), 0,
                                 stream, in, sig, kap, S, H, T);
    if (err != cudaSuccess) return err;
    return launch_fold(sig, kap, out, B, T, H, stream, dev);
}

int read_and_clear_device_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err, sizeof(v)) != cudaSuccess) return -1;
    if (v != 0 && cudaMemcpyToSymbol(g_err, &zero, sizeof(zero)) != cudaSuccess) return -1;
    return (int)v;
}

}  // namespace adaln

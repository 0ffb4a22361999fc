// Modulation projection 3072 -> 6144 (forward and backward).
//
// Operator: RL-Kernel PR 538 "final_adaln_out", section "What": scale, shift =
// (SiLU(temb) @ W^T + b).chunk(2), computed by a fixed-order projection and
// its backward.  At the batch sizes of a diffusion step (B = 1, 2) the work is
// weight-bandwidth bound (37.7 MB of W against B * 37.7 MFLOP), so every
// kernel here streams W once per call on CUDA cores, with an accumulation
// order that depends only on D, never on B or on a sample's position.
//
// Layout: W [2D, D] bf16 row-major (row n = output feature n), temb, u [B, D]
// bf16, emb [B, 2D] bf16, d_emb [B, 2D] fp32, dW [2D, D], db [2D].
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace adaln {

// --------------------------------------------------------------------------
// SiLU as a lookup: a bf16 input has 65536 values, so u = bf16(silu(t)) is
// tabulated once per device by silu_table_kernel (silu_bf16 on every bit
// pattern, the same bits as computing it in place).  silu_bf16 recomputes in
// fp64 near a bf16 rounding tie, and fp64 is slow on this GPU: one warp that
// takes that branch stalls for microseconds, so the hot kernels look the
// value up instead (128 KB, cached in L1 after first use).
// --------------------------------------------------------------------------
static __device__ uint16_t g_silu_tab[65536];

// device-side error word of this file's kernels (see adaln_device_error)
static __device__ unsigned g_err_proj;
__device__ __forceinline__ void report_error_proj(unsigned code) {
    if (code == kErrDrainFailed)
        atomicOr(&g_err_proj, code);
    else
        atomicCAS(&g_err_proj, 0u, code);
}

__global__ void __launch_bounds__(256) silu_table_kernel() {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < 65536) g_silu_tab[i] = silu_bf16((uint16_t)i);
}

// u for one packed bf16x2 word
__device__ __forceinline__ uint32_t silu_word(uint32_t w) {
    const uint32_t lo = __ldg(&g_silu_tab[w & 0xFFFFu]);
    const uint32_t hi = __ldg(&g_silu_tab[w >> 16]);
    return lo | (hi << 16);
}

// u = bf16(silu(temb)): 8 elements per thread
__global__ void __launch_bounds__(256) silu_kernel(const uint16_t *__restrict__ temb, uint16_t *__restrict__ u,
                                                   long long n8) {
    pdl_wait();
    pdl_trigger();  // the next kernel (the projection) reads u only after its own wait
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n8) return;
    const uint4 t = ldg16(temb + i * 8);
    stg16(u + i * 8, make_uint4(silu_word(t.x), silu_word(t.y), silu_word(t.z), silu_word(t.w)));
}

// --------------------------------------------------------------------------
// The projection's summation order, shared by both kernels below:
// emb[b,n] = bf16(sum_k u[b,k] W[n,k] + bias[n]), one warp per output row n.
// Lane l takes the 16-byte vectors v = l, l+32, l+64, ... of the row in
// ascending order; within a vector the element pairs (0,1), (2,3), (4,5),
// (6,7) in order, even elements into one fp32 accumulator and odd ones into
// another (one packed fused multiply-add per pair; each product of two bf16 is
// exact in fp32, so every term is rounded once).  Then the two accumulators are
// added, the lanes combine by a fixed xor butterfly, and the bias is added in
// fp32 before the one bf16 rounding.  The order depends on D only.
// --------------------------------------------------------------------------
__device__ __forceinline__ float2 dot_pairs(uint4 w, float2 u0, float2 u1, float2 u2, float2 u3, float2 acc) {
    acc = f2fma(u0, bf16x2_to_f2(w.x), acc);
    acc = f2fma(u1, bf16x2_to_f2(w.y), acc);
    acc = f2fma(u2, bf16x2_to_f2(w.z), acc);
    acc = f2fma(u3, bf16x2_to_f2(w.w), acc);
    return acc;
}

// emb for up to BC samples at a time; samples staged in shared memory as bf16.
constexpr int kFwdVL = 12;  // W vectors per lane held in registers (one row of D = 3072)

template <int BC>
__global__ void __launch_bounds__(256, 3)
proj_fwd_kernel(const uint16_t *__restrict__ W, const uint16_t *__restrict__ bias, const uint16_t *__restrict__ u,
                uint16_t *__restrict__ emb, int B, int D) {
    extern __shared__ __align__(128) uint4 us[];  // [BC][D/8]
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = 2 * D;
    const int V = D >> 3;
    const int n = blockIdx.x * 8 + warp;
    const bool live = n < N;
    const uint16_t *wrow = W + (size_t)(live ? n : N - 1) * D;
    const bool one_chunk = V <= 32 * kFwdVL;

    // W and bias are inputs of this call, never outputs of the kernel that
    // precedes this one (the SiLU kernel above), so they are read before the wait.
    uint4 wv[kFwdVL];
    const uint64_t pol_w = l2_evict_last();  // the backward projection reads W again
#pragma unroll
    for (int q = 0; q < kFwdVL; ++q) {
        const int v = lane + 32 * q;
        if (v < V) wv[q] = ldg16_hint(wrow + (size_t)v * 8, pol_w);
    }
    const float bn = bf16f(bias[live ? n : N - 1]);
    pdl_wait();

    for (int b0 = 0; b0 < B; b0 += BC) {
        const int nb = min(BC, B - b0);
        for (int i = threadIdx.x; i < nb * V; i += blockDim.x) us[i] = ldg16(u + (size_t)b0 * D + (size_t)i * 8);
        __syncthreads();
        float2 acc[BC];
#pragma unroll
        for (int b = 0; b < BC; ++b) acc[b] = make_float2(0.0f, 0.0f);
        for (int v0 = 0; v0 < V; v0 += 32 * kFwdVL) {
            if (!one_chunk && (v0 > 0 || b0 > 0)) {
#pragma unroll
                for (int q = 0; q < kFwdVL; ++q) {
                    const int v = v0 + lane + 32 * q;
                    if (v < V) wv[q] = ldg16_hint(wrow + (size_t)v * 8, pol_w);
                }
            }
#pragma unroll
            for (int q = 0; q < kFwdVL; ++q) {
                const int v = v0 + lane + 32 * q;
                if (v < V) {
#pragma unroll
                    for (int b = 0; b < BC; ++b) {
                        if (b < nb) {
                            const uint4 x = us[b * V + v];
                            acc[b] = dot_pairs(wv[q], bf16x2_to_f2(x.x), bf16x2_to_f2(x.y), bf16x2_to_f2(x.z),
                                               bf16x2_to_f2(x.w), acc[b]);
                        }
                    }
                }
            }
        }
#pragma unroll
        for (int b = 0; b < BC; ++b) {
            if (b < nb) {
                const float tot = warp_sum(__fadd_rn(acc[b].x, acc[b].y));
                if (lane == 0 && live) emb[(size_t)(b0 + b) * N + n] = bf16_bits(__fadd_rn(tot, bn));
            }
        }
        __syncthreads();
    }
    pdl_trigger();
}

// --------------------------------------------------------------------------
// The same projection for up to kStreamMaxB samples, after the SiLU kernel.
// W and bias are inputs of this call, and the kernel before this one is the
// SiLU kernel, which waits for all earlier work to complete before it lets
// this one start: the first W rows of every warp and the bias are loaded
// before this kernel's own wait, and stream in while SiLU runs.  Then u is
// staged in shared memory (fp32, two float4 planes per sample), and warp gw
// (global index, NW warps in all) takes rows n = gw, gw + NW, ..., two at a
// time for up to 2 samples (one otherwise), each lane holding its vectors
// v = lane + 32 j of the rows in registers.  The order of the terms is the
// one above, so both kernels give the same bits.
// --------------------------------------------------------------------------
constexpr int kStreamMaxB = 8;
constexpr int kStreamWarps = 8;
constexpr int kStreamVL = 12;  // W vectors per lane and row held in registers (D <= 3072)

template <int BC>
__global__ void __launch_bounds__(kStreamWarps * 32, 2)
proj_fwd_stream_kernel(const uint16_t *__restrict__ u, const uint16_t *__restrict__ W,
                       const uint16_t *__restrict__ bias, uint16_t *__restrict__ emb, int B, int D) {
    extern __shared__ __align__(128) float uf[];  // [B][D] fp32
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = 2 * D;
    const int V = D >> 3;

    const int NW = gridDim.x * kStreamWarps;
    const int gw = blockIdx.x * kStreamWarps + warp;
    const int nrows = gw < N ? (N - 1 - gw) / NW + 1 : 0;  // rows of this warp

    uint4 wa[kStreamVL], wb[kStreamVL];
    const uint64_t pol_w = l2_evict_last();  // the backward projection reads W again
    auto load_row = [&](uint4(&w)[kStreamVL], int n) {
#pragma unroll
        for (int j = 0; j < kStreamVL; ++j) {
            const int v = lane + 32 * j;
            w[j] = v < V ? ldg16_hint(W + (size_t)n * D + (size_t)v * 8, pol_w) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    constexpr int R = BC <= 2 ? 2 : 1;  // rows in flight per warp (registers)
    // the bias of this warp's rows (lane k holding row k, raw bits), then the first rows of W
    const uint16_t bias_raw = lane < nrows ? bias[gw + lane * NW] : (uint16_t)0;
    if (nrows > 0) load_row(wa, gw);
    if (R == 2 && nrows > 1) load_row(wb, gw + NW);
    pdl_wait();  // u comes from the SiLU kernel

    // u of every sample as fp32, per sample two planes of float4 (columns 0-3,
    // then 4-7 of every vector), so that the lanes of a warp read consecutive
    // 16-byte words
    for (int i = threadIdx.x; i < B * V; i += blockDim.x) {
        const uint4 t = ldg16(u + (size_t)i * 8);
        const int bi = i / V, vi = i - bi * V;
        float4 *dst = reinterpret_cast<float4 *>(uf + (size_t)bi * D);
        dst[vi] = make_float4(bf16lo(t.x), bf16hi(t.x), bf16lo(t.y), bf16hi(t.y));
        dst[V + vi] = make_float4(bf16lo(t.z), bf16hi(t.z), bf16lo(t.w), bf16hi(t.w));
    }
    __syncthreads();
    pdl_trigger();

    auto row_dot = [&](const uint4(&w)[kStreamVL], float2(&acc)[BC]) {
#pragma unroll
        for (int b = 0; b < BC; ++b) acc[b] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < kStreamVL; ++j) {
            const int v = lane + 32 * j;
            if (v < V) {
#pragma unroll
                for (int b = 0; b < BC; ++b) {
                    if (b < B) {
                        const float4 *up = reinterpret_cast<const float4 *>(uf + (size_t)b * D);
                        const float4 ua = up[v], ub = up[V + v];
                        acc[b] = dot_pairs(w[j], make_float2(ua.x, ua.y), make_float2(ua.z, ua.w),
                                           make_float2(ub.x, ub.y), make_float2(ub.z, ub.w), acc[b]);
                    }
                }
            }
        }
    };
    auto finish = [&](const float2(&acc)[BC], int k) {
        const int n = gw + k * NW;
        const float bk = bf16f((uint16_t)__shfl_sync(0xFFFFFFFFu, (uint32_t)bias_raw, k & 31));
        const float bn = k < 32 ? bk : bf16f(bias[n]);
#pragma unroll
        for (int b = 0; b < BC; ++b) {
            if (b < B) {
                const float tot = warp_sum(__fadd_rn(acc[b].x, acc[b].y));
                if (lane == 0) emb[(size_t)b * N + n] = bf16_bits(__fadd_rn(tot, bn));
            }
        }
    };
    if (R == 2) {
        for (int k = 0; k < nrows; k += 2) {
            float2 acc_a[BC], acc_b[BC];
            row_dot(wa, acc_a);
            if (k + 1 < nrows) row_dot(wb, acc_b);
            // the next two rows go in flight before the sums of these two
            if (k + 2 < nrows) load_row(wa, gw + (k + 2) * NW);
            if (k + 3 < nrows) load_row(wb, gw + (k + 3) * NW);
            finish(acc_a, k);
            if (k + 1 < nrows) finish(acc_b, k + 1);
        }
    } else {
        for (int k = 0; k < nrows; ++k) {
            float2 acc_a[BC];
            row_dot(wa, acc_a);
            if (k + 1 < nrows) load_row(wa, gw + (k + 1) * NW);
            finish(acc_a, k);
        }
    }
}

// --------------------------------------------------------------------------
// The projection for one or two samples (a diffusion step's batch) with all of
// W requested at once: one CTA per SM, each owning a contiguous range of about
// 2D / SMs rows.  Right after the dependency wait (and the small temb load),
// each of the 16 warps loads one row into registers, and the warps issue bulk
// copies of the CTA's other rows into shared memory (an mbarrier per copy), so
// the whole of W is in flight in one wave; meanwhile every CTA computes u = bf16(silu(temb))
// into shared memory (fp32, two float4 planes per sample).  Then each warp dots
// its register row, and the shared-memory rows as they land.  The order of the
// terms is the one above, so emb has the bits of the other kernels.
// --------------------------------------------------------------------------
constexpr int kWaveWarps = 16;
constexpr int kWaveMaxSmemRows = 32;
constexpr int kWaveChunkRows = 1;  // rows of W per bulk copy

// u = bf16(silu(t)) with the table's bits: computed in fp32 where the fp32 value
// is not near a bf16 rounding tie (the table holds that same value there), the
// table itself elsewhere
__device__ __forceinline__ uint32_t silu_fast(uint16_t tb) {
    const float t = bf16f(tb);
    if (t < -80.0f) return __ldg(&g_silu_tab[tb]);
    const float s = __fdiv_rn(t, __fadd_rn(1.0f, expf(-t)));
    const int low = (int)(__float_as_uint(s) & 0xFFFFu) - 0x8000;
    if (low <= 16 && low >= -16) return __ldg(&g_silu_tab[tb]);
    return bf16_bits(s);
}

template <int BC>
__global__ void __launch_bounds__(kWaveWarps * 32, 1)
proj_fwd_wave_kernel(const uint16_t *__restrict__ temb, const uint16_t *__restrict__ W,
                     const uint16_t *__restrict__ bias, uint16_t *__restrict__ emb, uint16_t *__restrict__ u_out,
                     int B, int D) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_raw);          // [chunks of rows]
    __shared__ int drain_needed;
    float *uf = reinterpret_cast<float *>(smem_raw + 256);            // [BC][D]
    unsigned char *wrows = smem_raw + 256 + (size_t)BC * D * 4;      // [rows][D] bf16
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = 2 * D;
    const int V = D >> 3;
    const int row_bytes = D * 2;
    const int r_begin = (int)(((long long)blockIdx.x * N) / gridDim.x);
    const int r_end = (int)(((long long)(blockIdx.x + 1) * N) / gridDim.x);
    const int nrows = r_end - r_begin;
    const int nreg = min(nrows, kWaveWarps);  // rows held in registers, one per warp
    const int nsm = nrows - nreg;             // rows staged in shared memory (the host checks the bound)

    if (threadIdx.x == 0) {
        for (int c = 0; c * kWaveChunkRows < nsm; ++c) mbar_init(&full[c], 1);
        drain_needed = 0;
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();  // temb, W and bias may come from the preceding kernel
    pdl_trigger();
    // temb first (12 KB per sample), so that it does not queue behind W
    constexpr int kTembPerThread = 2;  // B * D / 8 <= 768 vectors over 512 threads (the host checks)
    uint4 tv[kTembPerThread];
#pragma unroll
    for (int q = 0; q < kTembPerThread; ++q) {
        const int i = threadIdx.x + q * (int)blockDim.x;
        tv[q] = i < B * V ? ldg16(temb + (size_t)i * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
    const uint64_t pol_w = l2_evict_last();  // the backward projection reads W again
    // this warp's register row first (loads issued behind a burst of bulk
    // copies wait for it), then the shared-memory rows: consecutive rows of W,
    // so they go in copies of kWaveChunkRows rows, issued by different warps
    uint4 wr[kStreamVL];
    const bool has_reg = warp < nreg;
    const int nr = r_begin + warp;
#pragma unroll
    for (int j = 0; j < kStreamVL; ++j) {
        const int v = lane + 32 * j;
        wr[j] = (has_reg && v < V) ? ldg16_hint(W + (size_t)nr * D + (size_t)v * 8, pol_w) : make_uint4(0u, 0u, 0u, 0u);
    }
    const int nchunk = (nsm + kWaveChunkRows - 1) / kWaveChunkRows;
    if (lane == 0)
        for (int c = warp; c < nchunk; c += kWaveWarps) {
            const int i0 = c * kWaveChunkRows;
            const uint32_t bytes = (uint32_t)min(kWaveChunkRows, nsm - i0) * row_bytes;
            mbar_arrive_expect_tx(&full[c], bytes);
            bulk_g2s_hint(wrows + (size_t)i0 * row_bytes, W + (size_t)(r_begin + nreg + i0) * D, bytes, &full[c], pol_w);
        }
    // u of every sample as fp32 planes (columns 0-3, then 4-7 of every vector);
    // the first CTA also writes u out
#pragma unroll
    for (int q = 0; q < kTembPerThread; ++q) {
        const int i = threadIdx.x + q * (int)blockDim.x;
        if (i >= B * V) break;
        const uint4 t = tv[q];
        const uint32_t tw[4] = {t.x, t.y, t.z, t.w};
        uint32_t uw[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) uw[q] = silu_fast((uint16_t)(tw[q] & 0xFFFFu)) | (silu_fast((uint16_t)(tw[q] >> 16)) << 16);
        const int bi = i / V, vi = i - bi * V;
        float4 *dst = reinterpret_cast<float4 *>(uf + (size_t)bi * D);
        dst[vi] = make_float4(bf16lo(uw[0]), bf16hi(uw[0]), bf16lo(uw[1]), bf16hi(uw[1]));
        dst[V + vi] = make_float4(bf16lo(uw[2]), bf16hi(uw[2]), bf16lo(uw[3]), bf16hi(uw[3]));
        if (blockIdx.x == 0) stg16(u_out + (size_t)i * 8, make_uint4(uw[0], uw[1], uw[2], uw[3]));
    }
    __syncthreads();

    auto row_out = [&](const uint4(&w)[kStreamVL], int n) {
        float2 acc[BC];
#pragma unroll
        for (int b = 0; b < BC; ++b) acc[b] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int j = 0; j < kStreamVL; ++j) {
            const int v = lane + 32 * j;
            if (v < V) {
#pragma unroll
                for (int b = 0; b < BC; ++b) {
                    if (b < B) {
                        const float4 *up = reinterpret_cast<const float4 *>(uf + (size_t)b * D);
                        const float4 ua = up[v], ub = up[V + v];
                        acc[b] = dot_pairs(w[j], make_float2(ua.x, ua.y), make_float2(ua.z, ua.w),
                                           make_float2(ub.x, ub.y), make_float2(ub.z, ub.w), acc[b]);
                    }
                }
            }
        }
        const float bn = bf16f(bias[n]);
#pragma unroll
        for (int b = 0; b < BC; ++b) {
            if (b < B) {
                const float tot = warp_sum(__fadd_rn(acc[b].x, acc[b].y));
                if (lane == 0) emb[(size_t)b * N + n] = bf16_bits(__fadd_rn(tot, bn));
            }
        }
    };
    if (has_reg) row_out(wr, nr);
    for (int i = warp; i < nsm; i += kWaveWarps) {
        const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&full[i / kWaveChunkRows], 0u));
        if (!ok) {
            if (lane == 0) {
                report_error_proj(kErrProjFwdWait);
                drain_needed = 1;
            }
            break;
        }
        uint4 ws[kStreamVL];
        const uint4 *src = reinterpret_cast<const uint4 *>(wrows + (size_t)i * row_bytes);
#pragma unroll
        for (int j = 0; j < kStreamVL; ++j) {
            const int v = lane + 32 * j;
            ws[j] = v < V ? src[v] : make_uint4(0u, 0u, 0u, 0u);
        }
        row_out(ws, r_begin + nreg + i);
    }
    __syncthreads();
    if (drain_needed && threadIdx.x == 0)  // let every issued copy land before leaving
        for (int c = 0; c * kWaveChunkRows < nsm; ++c)
            if (!mbar_wait_bounded(&full[c], 0u, 10000000ull)) report_error_proj(kErrDrainFailed);
}

// --------------------------------------------------------------------------
// Backward, kernel 1: one CTA per (k-chunk of 256 columns, slab of 256 rows).
//
// Warp w takes the slab's rows n = n0 + w + 8 i (i ascending), lane l the 8
// columns k = k0 + 8 l .. +7; each warp keeps kPre rows of W in flight.  For
// the samples of the current chunk it adds e[b,n] * W[n,k] into fp32 partials
// (each product exact), then the 8 warps' partials are added in ascending warp
// order and written per slab: ws[slab][b][k].  The slab size, and so this
// order, depends on D only.  With WITH_W (all samples in one chunk) it also
// produces dW and db for its tile: acc = (accumulate ? acc_in : +0), then
// + e[b,n] * u[b,k] for b ascending, one rounding per add.
// --------------------------------------------------------------------------
constexpr int kSlabRows = kProjSlabRows;        // 256
constexpr int kRowsPerWarp = kSlabRows / 8;     // 32
constexpr int kPreMax = 8;                       // rows of W per register batch (two batches, up to 2 samples)

template <int BC>
struct SlabSmem {
    float es[BC][kSlabRows];
    float red[8][BC][kProjKChunk];
};

// What the slab kernel writes besides the d_silu partials (a template
// argument, so the per-row loop carries no runtime branches):
//   kSlabDsOnly   nothing (dW and db come from the tiled kernels)
//   kSlabDwOut    dW and db in bf16, overwrite, no fp32 accumulators
//   kSlabGeneral  any of dW_acc, db_acc (accumulate or overwrite), dW, db
//   kSlabDwFull   kSlabDwOut where every slab is whole (D % 256 == 0, so every
//                 warp has 32 rows and every lane's columns lie inside D) and
//                 the chunk holds all BC samples: no per-row tests, row
//                 pointers stepped by a fixed stride, db after the rows
constexpr int kSlabDsOnly = 0, kSlabDwOut = 1, kSlabGeneral = 2, kSlabDwFull = 3;

template <int BC, int WM>
__global__ void __launch_bounds__(256, 2)
proj_bwd_slab_kernel(const float *__restrict__ d_emb, const uint16_t *__restrict__ u, const uint16_t *__restrict__ W,
                     float *__restrict__ dW_acc, float *__restrict__ db_acc, uint16_t *__restrict__ dW,
                     uint16_t *__restrict__ db, int accumulate, float *__restrict__ ws, int B, int D) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    SlabSmem<BC> &sm = *reinterpret_cast<SlabSmem<BC> *>(smem_raw);
    constexpr bool WITH_W = WM != kSlabDsOnly;
    const int kchunk = blockIdx.x;
    const int slab = blockIdx.y;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = 2 * D;
    const int n0 = slab * kSlabRows;
    const int kv = kchunk * 32 + lane;
    const bool live_k = kv < (D >> 3);
    const int col = kv * 8;
    const int cnt = min(kRowsPerWarp, (N - n0) / 8);  // rows per warp, equal for all warps (N % 16 == 0)
    const bool want_dw = WM == kSlabDwOut || (WM == kSlabGeneral && (dW_acc != nullptr || dW != nullptr));
    const bool want_db = (WM == kSlabDwOut || (WM == kSlabGeneral && (db_acc != nullptr || db != nullptr))) &&
                         kchunk == 0 && lane == 0;
    constexpr int kPre = BC <= 2 ? kPreMax : kPreMax / 2;  // fewer rows in flight where more samples need registers

    // W is an input of this call: its rows of this CTA are brought into L2
    // while the preceding kernel finishes (L2 is the point of coherence, so
    // reads after the wait still see any write of the preceding kernel)
    if (B > 0 && threadIdx.x < kSlabRows && n0 + (int)threadIdx.x < N && kchunk * kProjKChunk < D)
        bulk_prefetch_l2(W + (size_t)(n0 + threadIdx.x) * D + (size_t)kchunk * kProjKChunk,
                         (uint32_t)min(kProjKChunk, D - kchunk * kProjKChunk) * 2u);
    pdl_wait();
    pdl_trigger();  // the next kernel may become resident and wait for this one
    const uint64_t pol_dw = l2_evict_first();  // dW is written once

    for (int b0 = 0; b0 < B || (WITH_W && b0 == 0); b0 += BC) {
        const int nb = max(0, min(BC, B - b0));
        for (int i = threadIdx.x; i < BC * kSlabRows; i += blockDim.x) {
            const int b = i / kSlabRows, r = i % kSlabRows;
            const int n = n0 + r;
            sm.es[b][r] = (b < nb && n < N) ? bf16f(bf16_bits(d_emb[(size_t)(b0 + b) * N + n])) : 0.0f;
        }
        float2 uf[BC][4];  // u of this lane's 8 columns, by column pair
#pragma unroll
        for (int b = 0; b < BC; ++b) {
            const uint4 uv = (WITH_W && b < nb && live_k) ? ldg16(u + (size_t)(b0 + b) * D + col) : make_uint4(0u, 0u, 0u, 0u);
            uf[b][0] = bf16x2_to_f2(uv.x); uf[b][1] = bf16x2_to_f2(uv.y);
            uf[b][2] = bf16x2_to_f2(uv.z); uf[b][3] = bf16x2_to_f2(uv.w);
        }
        __syncthreads();

        // d_silu partials of this lane's columns, by column pair (each lane of a
        // packed operation is one column, in its own sequential order)
        float2 ds[BC][4];
#pragma unroll
        for (int b = 0; b < BC; ++b)
#pragma unroll
            for (int q = 0; q < 4; ++q) ds[b][q] = make_float2(0.0f, 0.0f);

        // W rows in two register batches of kPre, double-buffered: one batch is
        // in flight while the other is used
        uint4 wa[kPre], wb[kPre];
        auto load_batch = [&](uint4(&wv)[kPre], int i0) {
#pragma unroll
            for (int p = 0; p < kPre; ++p) {
                const int n = n0 + warp + 8 * (i0 + p);
                wv[p] = make_uint4(0u, 0u, 0u, 0u);  // W is not read without samples
                if (i0 + p < cnt && live_k && nb > 0) wv[p] = ldg16(W + (size_t)n * D + col);
            }
        };
        auto use_batch = [&](const uint4(&wv)[kPre], int i0) {
#pragma unroll
            for (int p = 0; p < kPre; ++p) {
                const int i = i0 + p;
                if (i < cnt && live_k) {
                    const int r = warp + 8 * i;
                    const int n = n0 + r;
                    const float2 w2[4] = {bf16x2_to_f2(wv[p].x), bf16x2_to_f2(wv[p].y), bf16x2_to_f2(wv[p].z),
                                          bf16x2_to_f2(wv[p].w)};
                    float2 e2[BC];
#pragma unroll
                    for (int b = 0; b < BC; ++b) e2[b] = f2splat(sm.es[b][r]);
#pragma unroll
                    for (int b = 0; b < BC; ++b)
                        if (b < nb) {
#pragma unroll
                            for (int q = 0; q < 4; ++q) ds[b][q] = f2fma(e2[b], w2[q], ds[b][q]);
                        }
                    if (WITH_W && want_dw) {
                        // acc = (accumulate ? acc_in : +0), then + e[b,n] * u[b,k] for b ascending
                        float2 acc[4];
                        float *pa = (WM == kSlabGeneral && dW_acc) ? dW_acc + (size_t)n * D + col : nullptr;
                        if (WM == kSlabGeneral && accumulate) {
                            const float4 a0 = *reinterpret_cast<const float4 *>(pa);
                            const float4 a1 = *reinterpret_cast<const float4 *>(pa + 4);
                            acc[0] = make_float2(a0.x, a0.y); acc[1] = make_float2(a0.z, a0.w);
                            acc[2] = make_float2(a1.x, a1.y); acc[3] = make_float2(a1.z, a1.w);
                        } else {
#pragma unroll
                            for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.0f, 0.0f);
                        }
#pragma unroll
                        for (int b = 0; b < BC; ++b)
                            if (b < nb) {
#pragma unroll
                                for (int q = 0; q < 4; ++q) acc[q] = f2fma(e2[b], uf[b][q], acc[q]);
                            }
                        if (WM == kSlabGeneral && pa) {
                            stg16f(pa, make_float4(acc[0].x, acc[0].y, acc[1].x, acc[1].y));
                            stg16f(pa + 4, make_float4(acc[2].x, acc[2].y, acc[3].x, acc[3].y));
                        }
                        if (WM == kSlabDwOut || dW)
                            stg16_hint(dW + (size_t)n * D + col,
                                       make_uint4(pack_bf16x2(acc[0].x, acc[0].y), pack_bf16x2(acc[1].x, acc[1].y),
                                                  pack_bf16x2(acc[2].x, acc[2].y), pack_bf16x2(acc[3].x, acc[3].y)),
                                       pol_dw);
                    }
                }
                if (WITH_W && want_db && i < cnt) {
                    const int r = warp + 8 * i;
                    const int n = n0 + r;
                    float a = (WM == kSlabGeneral && accumulate) ? db_acc[n] : 0.0f;
                    for (int b = 0; b < nb; ++b) a = __fadd_rn(a, sm.es[b][r]);
                    if (WM == kSlabGeneral && db_acc) db_acc[n] = a;
                    if (WM == kSlabDwOut || db) db[n] = bf16_bits(a);
                }
            }
        };
        // kSlabDwFull: the same arithmetic in the same order as kSlabDwOut
        if constexpr (WM == kSlabDwFull) {
            const size_t step = (size_t)8 * D;  // from one of this warp's rows to the next
            const uint16_t *wrow = W + (size_t)(n0 + warp) * D + col;
            uint16_t *drow = dW + (size_t)(n0 + warp) * D + col;
            auto fload = [&](uint4(&wv)[kPre], int i0) {
#pragma unroll
                for (int p = 0; p < kPre; ++p) wv[p] = ldg16(wrow + (size_t)(i0 + p) * step);
            };
            auto fuse = [&](const uint4(&wv)[kPre], int i0) {
#pragma unroll
                for (int p = 0; p < kPre; ++p) {
                    const int r = warp + 8 * (i0 + p);
                    const float2 w2[4] = {bf16x2_to_f2(wv[p].x), bf16x2_to_f2(wv[p].y), bf16x2_to_f2(wv[p].z),
                                          bf16x2_to_f2(wv[p].w)};
                    float2 acc[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc[q] = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int b = 0; b < BC; ++b) {
                        const float2 e2 = f2splat(sm.es[b][r]);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            ds[b][q] = f2fma(e2, w2[q], ds[b][q]);
                            acc[q] = f2fma(e2, uf[b][q], acc[q]);
                        }
                    }
                    stg16_hint(drow + (size_t)(i0 + p) * step,
                               make_uint4(pack_bf16x2(acc[0].x, acc[0].y), pack_bf16x2(acc[1].x, acc[1].y),
                                          pack_bf16x2(acc[2].x, acc[2].y), pack_bf16x2(acc[3].x, acc[3].y)),
                               pol_dw);
                }
            };
            fload(wa, 0);
            fload(wb, kPre);
#pragma unroll
            for (int i0 = 0; i0 < kRowsPerWarp; i0 += 2 * kPre) {
                fuse(wa, i0);
                if (i0 + 2 * kPre < kRowsPerWarp) fload(wa, i0 + 2 * kPre);
                fuse(wb, i0 + kPre);
                if (i0 + 3 * kPre < kRowsPerWarp) fload(wb, i0 + 3 * kPre);
            }
            // db of the slab's rows: samples in ascending order from +0, one thread per row
            if (kchunk == 0)
                for (int rr = threadIdx.x; rr < kSlabRows; rr += blockDim.x) {
                    float a = 0.0f;
                    for (int b = 0; b < nb; ++b) a = __fadd_rn(a, sm.es[b][rr]);
                    db[n0 + rr] = bf16_bits(a);
                }
        } else {
            load_batch(wa, 0);
            load_batch(wb, kPre);
            for (int i0 = 0; i0 < cnt; i0 += 2 * kPre) {
                use_batch(wa, i0);
                if (i0 + 2 * kPre < cnt) load_batch(wa, i0 + 2 * kPre);
                use_batch(wb, i0 + kPre);
                if (i0 + 3 * kPre < cnt) load_batch(wb, i0 + 3 * kPre);
            }
        }
        // the slab's partial d_silu: warps added in ascending order
#pragma unroll
        for (int b = 0; b < BC; ++b) {
            float4 *dst = reinterpret_cast<float4 *>(&sm.red[warp][b][lane * 8]);
            dst[0] = make_float4(ds[b][0].x, ds[b][0].y, ds[b][1].x, ds[b][1].y);
            dst[1] = make_float4(ds[b][2].x, ds[b][2].y, ds[b][3].x, ds[b][3].y);
        }
        __syncthreads();
        for (int i = threadIdx.x; i < nb * kProjKChunk; i += blockDim.x) {
            const int b = i / kProjKChunk, c = i % kProjKChunk;
            const int k = kchunk * kProjKChunk + c;
            if (k < D) {
                float tot = sm.red[0][b][c];
#pragma unroll
                for (int w = 1; w < 8; ++w) tot = __fadd_rn(tot, sm.red[w][b][c]);
                __stcg(ws + ((size_t)slab * B + b0 + b) * D + k, tot);
            }
        }
        __syncthreads();
    }
}

// --------------------------------------------------------------------------
// Backward, kernel 2: d_temb[b,k] = bf16((sum over slabs, ascending) * silu'(t))
// --------------------------------------------------------------------------
constexpr int kMaxSlabs = 2 * kMaxD / kProjSlabRows;  // 64

__global__ void __launch_bounds__(256)
proj_bwd_final_kernel(const float *__restrict__ ws, const uint16_t *__restrict__ temb, uint16_t *__restrict__ d_temb,
                      int B, int D, int nslab) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long BD = (long long)B * D;
    // silu'(t) before the wait: temb is an input of this call, the kernels
    // before this one are the call's own (they cannot write temb: outputs
    // never overlap inputs), and the call's first kernel let this one start
    // only after its own wait, i.e. after all earlier work had completed
    const float ds = i < BD ? dsilu_f32(bf16f(temb[i])) : 0.0f;
    pdl_wait();
    pdl_trigger();
    if (i < BD) {
        float tot;
        if (nslab == 24) {
            // D = 3072: all 24 partials requested before the first add
            float part[24];
#pragma unroll
            for (int s = 0; s < 24; ++s) part[s] = __ldcg(ws + (size_t)s * BD + i);
            tot = part[0];
#pragma unroll
            for (int s = 1; s < 24; ++s) tot = __fadd_rn(tot, part[s]);
        } else {
            // all partials are loaded before the first add (nslab <= kMaxSlabs)
            float part[kMaxSlabs];
#pragma unroll
            for (int s = 0; s < kMaxSlabs; ++s) part[s] = s < nslab ? __ldcg(ws + (size_t)s * BD + i) : 0.0f;
            tot = part[0];
#pragma unroll
            for (int s = 1; s < kMaxSlabs; ++s)
                if (s < nslab) tot = __fadd_rn(tot, part[s]);
        }
        d_temb[i] = bf16_bits(__fmul_rn(tot, ds));
    }
}

// --------------------------------------------------------------------------
// dW for many samples: a 128 x 128 tile of dW per CTA, thread (tn, tk) owning
// rows r0 + 8 tn .. +7 and columns k0 + 8 tk .. +7 (64 accumulators: 64
// fused multiply-adds per 4 shared-memory loads of a sample); samples stream
// through shared memory 16 at a time and are added in ascending order,
// exactly as in the slab kernel: acc = acc + e[b,n] * u[b,k].
// --------------------------------------------------------------------------
constexpr int kDwTile = 128;
constexpr int kDwBChunk = 16;

__global__ void __launch_bounds__(256, 2)
proj_dw_tiled_kernel(const float *__restrict__ d_emb, const uint16_t *__restrict__ u, float *__restrict__ dW_acc,
                     uint16_t *__restrict__ dW, int accumulate, int B, int D, int n_begin, int nrows) {
    // rows n_begin .. n_begin + nrows - 1 of the gradient; outputs indexed from that first row
    __shared__ __align__(16) float es[kDwBChunk][kDwTile];
    __shared__ __align__(16) float us[kDwBChunk][kDwTile];
    const int N = 2 * D;
    const int k0 = blockIdx.x * kDwTile;
    const int r0 = blockIdx.y * kDwTile;  // first output row of the tile, relative to n_begin
    const int tk = threadIdx.x & 15;
    const int tn = threadIdx.x >> 4;
    pdl_wait();
    pdl_trigger();
    float acc[8][8];
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int r = r0 + 8 * tn + a;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const int k = k0 + 8 * tk + c;
            acc[a][c] = (accumulate && r < nrows && k < D) ? dW_acc[(size_t)r * D + k] : 0.0f;
        }
    }
    for (int b0 = 0; b0 < B; b0 += kDwBChunk) {
        const int nb = min(kDwBChunk, B - b0);
        for (int i = threadIdx.x; i < kDwBChunk * kDwTile; i += blockDim.x) {
            const int b = i / kDwTile, j = i % kDwTile;
            const int r = r0 + j, k = k0 + j;
            es[b][j] = (b < nb && r < nrows) ? bf16f(bf16_bits(d_emb[(size_t)(b0 + b) * N + n_begin + r])) : 0.0f;
            us[b][j] = (b < nb && k < D) ? bf16f(u[(size_t)(b0 + b) * D + k]) : 0.0f;
        }
        __syncthreads();
        for (int b = 0; b < nb; ++b) {
            const float4 e0 = *reinterpret_cast<const float4 *>(&es[b][8 * tn]);
            const float4 e1 = *reinterpret_cast<const float4 *>(&es[b][8 * tn + 4]);
            const float4 u0 = *reinterpret_cast<const float4 *>(&us[b][8 * tk]);
            const float4 u1 = *reinterpret_cast<const float4 *>(&us[b][8 * tk + 4]);
            const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
            const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
            for (int a = 0; a < 8; ++a)
#pragma unroll
                for (int c = 0; c < 8; ++c) acc[a][c] = __fmaf_rn(ev[a], uv[c], acc[a][c]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 8; ++a) {
        const int r = r0 + 8 * tn + a;
        const int k = k0 + 8 * tk;
        if (r < nrows && k < D) {  // D % 8 == 0, so the 8 columns are all in range
            if (dW_acc) {
                stg16f(dW_acc + (size_t)r * D + k, make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]));
                stg16f(dW_acc + (size_t)r * D + k + 4, make_float4(acc[a][4], acc[a][5], acc[a][6], acc[a][7]));
            }
            if (dW)
                stg16(dW + (size_t)r * D + k,
                      make_uint4(pack_bf16x2(acc[a][0], acc[a][1]), pack_bf16x2(acc[a][2], acc[a][3]),
                                 pack_bf16x2(acc[a][4], acc[a][5]), pack_bf16x2(acc[a][6], acc[a][7])));
        }
    }
}

__global__ void __launch_bounds__(256)
proj_db_kernel(const float *__restrict__ d_emb, float *__restrict__ db_acc, uint16_t *__restrict__ db, int accumulate,
               int B, int N, int n_begin, int nrows) {
    pdl_wait();
    pdl_trigger();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < nrows) {
        float a = accumulate ? db_acc[r] : 0.0f;
        for (int b = 0; b < B; ++b) a = __fadd_rn(a, bf16f(bf16_bits(d_emb[(size_t)b * N + n_begin + r])));
        if (db_acc) db_acc[r] = a;
        if (db) db[r] = bf16_bits(a);
    }
}

// --------------------------------------------------------------------------
// launchers
// --------------------------------------------------------------------------
template <int BC>
static cudaError_t launch_proj_fwd_gemv(const uint16_t *W, const uint16_t *bias, const uint16_t *u, uint16_t *emb,
                                        int B, int D, cudaStream_t stream, const DeviceInfo &dev) {
    const size_t smem = (size_t)BC * D * 2;
    auto kern = proj_fwd_kernel<BC>;
    cudaError_t err = ensure_smem_attr((const void *)kern, smem, dev);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3((2 * D + 7) / 8), dim3(256), smem, stream, W, bias, u, emb, B, D);
}

template <int BC>
static cudaError_t launch_proj_fwd_stream(const uint16_t *u, const uint16_t *W, const uint16_t *bias, uint16_t *emb,
                                          int B, int D, size_t smem, cudaStream_t stream, const DeviceInfo &dev) {
    auto kern = proj_fwd_stream_kernel<BC>;
    cudaError_t err = ensure_smem_attr((const void *)kern, smem, dev);
    if (err != cudaSuccess) return err;
    int per_sm = 0;
    err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kStreamWarps * 32, smem);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) per_sm = 1;
    const int N = 2 * D;
    int grid = dev.sm_count * per_sm;
    const int need = (N + kStreamWarps - 1) / kStreamWarps;
    if (grid > need) grid = need;
    return launch_pdl(kern, dim3(grid), dim3(kStreamWarps * 32), smem, stream, u, W, bias, emb, B, D);
}

// The SiLU table of the current device, filled by its first call: launched on
// the caller's stream, which is then synchronized once, so that calls on other
// streams never read the table before it is complete.
static std::mutex g_tab_mu;
static bool g_tab_ready[64];

static cudaError_t ensure_silu_table(cudaStream_t stream, const DeviceInfo &dev) {
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_tab_mu);
    if (g_tab_ready[dev.device]) return cudaSuccess;
    silu_table_kernel<<<65536 / 256, 256, 0, stream>>>();
    cudaError_t err = cudaGetLastError();
    if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
    if (err == cudaSuccess) g_tab_ready[dev.device] = true;
    return err;
}

template <int BC>
static cudaError_t launch_proj_fwd_wave(const uint16_t *temb, const uint16_t *W, const uint16_t *bias, uint16_t *emb,
                                        uint16_t *u, int B, int D, size_t smem, cudaStream_t stream,
                                        const DeviceInfo &dev) {
    auto kern = proj_fwd_wave_kernel<BC>;
    cudaError_t err = ensure_smem_attr((const void *)kern, smem, dev);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(dev.sm_count), dim3(kWaveWarps * 32), smem, stream, temb, W, bias, emb, u, B, D);
}

// D a multiple of 64: the SiLU kernel, then the tensor-core projection
// (tc_proj.cu), for every B.  Other D (one order of the CUDA-core kernels for
// every B): one or two samples with D <= 3072 (when every SM can hold its
// share of W), the one-wave kernel; otherwise the SiLU kernel, then up to
// kStreamMaxB samples and D <= 3072 the streaming GEMV, else the chunked GEMV.
cudaError_t launch_proj_fwd(const uint16_t *temb, const uint16_t *W, const uint16_t *bias, uint16_t *emb,
                            uint16_t *u, int B, int D, cudaStream_t stream, const DeviceInfo &dev) {
    if (B == 0) return cudaSuccess;
    cudaError_t err = ensure_silu_table(stream, dev);
    if (err != cudaSuccess) return err;
    if (proj_fwd_tc_supported(D)) {
        const long long n8 = (long long)B * D / 8;
        err = launch_pdl(silu_kernel, dim3((unsigned)((n8 + 255) / 256)), dim3(256), 0, stream, temb, u, n8);
        if (err != cudaSuccess) return err;
        return launch_proj_fwd_tc(u, W, bias, emb, B, D, stream, dev);
    }
    if (B <= 2 && D / 8 <= 32 * kStreamVL && dev.sm_count > 0 && B * (D / 8) <= 2 * kWaveWarps * 32) {
        const int N = 2 * D;
        const int rows_max = (N + dev.sm_count - 1) / dev.sm_count;
        const int nsm_max = rows_max > kWaveWarps ? rows_max - kWaveWarps : 0;
        const size_t smem = 256 + (size_t)(B == 1 ? 1 : 2) * D * 4 + (size_t)nsm_max * D * 2;
        if (nsm_max <= kWaveMaxSmemRows && smem <= 227 * 1024) {
            if (B == 1) return launch_proj_fwd_wave<1>(temb, W, bias, emb, u, B, D, smem, stream, dev);
            return launch_proj_fwd_wave<2>(temb, W, bias, emb, u, B, D, smem, stream, dev);
        }
    }
    const long long n8 = (long long)B * D / 8;
    err = launch_pdl(silu_kernel, dim3((unsigned)((n8 + 255) / 256)), dim3(256), 0, stream, temb, u, n8);
    if (err != cudaSuccess) return err;
    if (B <= kStreamMaxB && D / 8 <= 32 * kStreamVL) {
        const size_t smem = (size_t)B * D * 4;
        if (B == 1) return launch_proj_fwd_stream<1>(u, W, bias, emb, B, D, smem, stream, dev);
        if (B == 2) return launch_proj_fwd_stream<2>(u, W, bias, emb, B, D, smem, stream, dev);
        if (B <= 4) return launch_proj_fwd_stream<4>(u, W, bias, emb, B, D, smem, stream, dev);
        return launch_proj_fwd_stream<8>(u, W, bias, emb, B, D, smem, stream, dev);
    }
    if (B <= 4) return launch_proj_fwd_gemv<4>(W, bias, u, emb, B, D, stream, dev);
    return launch_proj_fwd_gemv<8>(W, bias, u, emb, B, D, stream, dev);
}


template <int BC, int WM>
static cudaError_t launch_slab(const float *d_emb, const uint16_t *u, const uint16_t *W, float *dW_acc, float *db_acc,
                               uint16_t *dW, uint16_t *db, int accumulate, float *ws, int B, int D,
                               cudaStream_t stream, const DeviceInfo &dev) {
    const size_t smem = sizeof(SlabSmem<BC>);
    auto kern = proj_bwd_slab_kernel<BC, WM>;
    cudaError_t err = ensure_smem_attr((const void *)kern, smem, dev);
    if (err != cudaSuccess) return err;
    const int nslab = (2 * D + kSlabRows - 1) / kSlabRows;
    const int nk = (D + kProjKChunk - 1) / kProjKChunk;
    return launch_pdl(kern, dim3(nk, nslab), dim3(256), smem, stream, d_emb, u, W, dW_acc, db_acc, dW, db,
                      accumulate, ws, B, D);
}

template <int BC>
static cudaError_t launch_slab_w(const float *d_emb, const uint16_t *u, const uint16_t *W, float *dW_acc,
                                 float *db_acc, uint16_t *dW, uint16_t *db, int accumulate, float *ws, int B, int D,
                                 cudaStream_t stream, const DeviceInfo &dev) {
    // dW and db both wanted in bf16, nothing accumulated: the branch-free form
    if (!dW_acc && !db_acc && !accumulate && dW && db) {
        if (D % kProjKChunk == 0 && B == BC)
            return launch_slab<BC, kSlabDwFull>(d_emb, u, W, dW_acc, db_acc, dW, db, accumulate, ws, B, D, stream,
                                                dev);
        return launch_slab<BC, kSlabDwOut>(d_emb, u, W, dW_acc, db_acc, dW, db, accumulate, ws, B, D, stream, dev);
    }
    return launch_slab<BC, kSlabGeneral>(d_emb, u, W, dW_acc, db_acc, dW, db, accumulate, ws, B, D, stream, dev);
}

// dW and db of the output rows [n0, n1) over all B samples (ascending), by the
// tiled kernels; outputs indexed from row n0
cudaError_t launch_wgrad_rows(const float *d_emb, const uint16_t *u, int n0, int n1, float *dW_acc, float *db_acc,
                              uint16_t *dW, uint16_t *db, int accumulate, int B, int D, cudaStream_t stream) {
    const int N = 2 * D;
    const int nrows = n1 - n0;
    cudaError_t err = cudaSuccess;
    if (nrows <= 0) return err;
    if (dW_acc || dW)
        err = launch_pdl(proj_dw_tiled_kernel, dim3((D + kDwTile - 1) / kDwTile, (nrows + kDwTile - 1) / kDwTile),
                         dim3(256), 0, stream, d_emb, u, dW_acc, dW, accumulate, B, D, n0, nrows);
    if (err == cudaSuccess && (db_acc || db))
        err = launch_pdl(proj_db_kernel, dim3((nrows + 255) / 256), dim3(256), 0, stream, d_emb, db_acc, db, accumulate,
                         B, N, n0, nrows);
    return err;
}

cudaError_t launch_proj_bwd(const float *d_emb, const uint16_t *temb, const uint16_t *u, const uint16_t *W,
                            uint16_t *d_temb, float *dW_acc, float *db_acc, uint16_t *dW, uint16_t *db,
                            int accumulate, void *ws_v, int B, int D, cudaStream_t stream, const DeviceInfo &dev) {
    float *ws = static_cast<float *>(ws_v);
    const int N = 2 * D;
    const int nslab = (N + kSlabRows - 1) / kSlabRows;
    cudaError_t err;
    if (B <= 4) {
        // one pass over W: d_silu partials and (when asked) dW / db
        if (B <= 1) err = launch_slab_w<1>(d_emb, u, W, dW_acc, db_acc, dW, db, accumulate, ws, B, D, stream, dev);
        else if (B == 2) err = launch_slab_w<2>(d_emb, u, W, dW_acc, db_acc, dW, db, accumulate, ws, B, D, stream, dev);
        else err = launch_slab_w<4>(d_emb, u, W, dW_acc, db_acc, dW, db, accumulate, ws, B, D, stream, dev);
    } else {
        err = launch_slab<4, kSlabDsOnly>(d_emb, u, W, nullptr, nullptr, nullptr, nullptr, 0, ws, B, D, stream, dev);
        if (err == cudaSuccess) err = launch_wgrad_rows(d_emb, u, 0, N, dW_acc, db_acc, dW, db, accumulate, B, D, stream);
    }
    if (err != cudaSuccess || B == 0) return err;
    const long long BD = (long long)B * D;
    return launch_pdl(proj_bwd_final_kernel, dim3((unsigned)((BD + 255) / 256)), dim3(256), 0, stream, ws, temb,
                      d_temb, B, D, nslab);
}

int read_and_clear_proj_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_proj, sizeof(v)) != cudaSuccess) return -1;
    if (v != 0 && cudaMemcpyToSymbol(g_err_proj, &zero, sizeof(zero)) != cudaSuccess) return -1;
    return (int)v;
}

}  // namespace adaln

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
// a copy that did not land within the drain's limit while a kernel was leaving
// after an error: marked by a bit of its own next to the first error code
__device__ __forceinline__ void report_drain_failure() { atomicOr(&g_err, kErrDrainFailed); }
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
    if (!mbar_wait_bounded(bar, parity, 10000000ull)) report_drain_failure();
}

// Test builds only (ADALN_TEST_WAIT_NEVER_NS defined): the first wait of each
// waiting warp goes to an mbarrier that nothing ever arrives on, with that
// limit in nanoseconds, so the time-out path (error word, drain of the issued
// copies, early return) runs on the GPU without any fault or hang.  Release
// builds compile none of it.
#ifdef ADALN_TEST_WAIT_NEVER_NS
#define ADALN_NEVER_BAR uint64_t never;
__device__ __forceinline__ bool test_wait_never(uint64_t *never) {
    return mbar_wait_bounded(never, 0u, (uint64_t)(ADALN_TEST_WAIT_NEVER_NS));
}
#else
#define ADALN_NEVER_BAR
#endif

// ==========================================================================
// Forward: one warp-group (128 threads) per token row, persistent.
//
// A CTA holds kWG warp-groups; each owns a contiguous range of rows and a ring
// of kFwdStages row buffers in shared memory, filled by 1-D bulk copies (the
// TMA engine).  Rows are taken in blocks of kFwdBlock: the row sums of the
// block, one barrier, the means; the sums of squared deviations, one barrier,
// the rstd values; then the outputs, recomputed from the staged rows, and a
// barrier that frees the block's stages for refilling.  Thread t of a
// warp-group owns the 16-byte vectors v = t + 128 j (8 columns each), so its
// modulation parameters stay in registers while the sample is unchanged.  The
// reduction order over d: per thread in (j, column pair) order, the two halves
// of the pairs, a fixed xor butterfly within the warp, then the four warps in
// ascending order.  It depends on D only.
// ==========================================================================
constexpr int kWG = 2;          // warp-groups per CTA
constexpr int kFwdBlock = 4;    // most rows per block (a block of BLK rows, NST = 2 BLK stages:
                                // two blocks in flight per warp-group)

struct FwdSmem {
    float red[kWG][2][kFwdBlock][4];  // [warp-group][sum, squares][row of block][warp]
    float mu[kWG][kFwdBlock], rs[kWG][kFwdBlock];
    uint64_t full[kWG][2 * kFwdBlock];
    ADALN_NEVER_BAR
};

// barrier of one warp-group, and a vote: is `flag` set in any of its threads?
__device__ __forceinline__ bool wg_barrier_or(int id, bool flag) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((unsigned)flag), "r"(id)
        : "memory");
    return r != 0;
}

template <int VPT, int BLK, int NST, int MINB>
__global__ void __launch_bounds__(kWG * 128, MINB)
out_fwd_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ emb, uint16_t *__restrict__ out,
               float *__restrict__ mean, float *__restrict__ rstd, int S, int D, float eps, long long R,
               int keep_out) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    FwdSmem &sm = *reinterpret_cast<FwdSmem *>(smem_raw);
    const int row_bytes = D * 2;
    unsigned char *stages = smem_raw + ((sizeof(FwdSmem) + 127) / 128) * 128;

    const int wg = threadIdx.x >> 7;
    const int t = threadIdx.x & 127;
    const int warp = t >> 5;
    const int lane = t & 31;
    const int V = D >> 3;
    unsigned char *my_stages = stages + (size_t)wg * NST * row_bytes;

    const long long G = (long long)gridDim.x * kWG;
    const long long g = (long long)blockIdx.x * kWG + wg;
    const long long r_begin = (g * R) / G;
    const long long r_end = ((g + 1) * R) / G;
    const int nrows = (int)(r_end - r_begin);

    if (t == 0) {
        for (int s = 0; s < NST; ++s) mbar_init(&sm.full[wg][s], 1);
#ifdef ADALN_TEST_WAIT_NEVER_NS
        if (wg == 0) mbar_init(&sm.never, 1);
#endif
        fence_barrier_init();
        // warm L2 with the first rows while the preceding kernel finishes
        for (int i = 0; i < NST && i < nrows; ++i) bulk_prefetch_l2(x + (size_t)(r_begin + i) * D, row_bytes);
    }
    __syncthreads();
    pdl_wait();  // inputs may come from the preceding kernel: read them only now
    pdl_trigger();

    if (t == 0)
        for (int i = 0; i < NST && i < nrows; ++i) {
            mbar_arrive_expect_tx(&sm.full[wg][i], row_bytes);
            bulk_g2s(my_stages + (size_t)i * row_bytes, x + (size_t)(r_begin + i) * D, row_bytes, &sm.full[wg][i]);
        }

    float2 onep[VPT][4], shift[VPT][4];  // modulation parameters of the current sample, by column pair
    long long cur_b = -1;
    const float Df = (float)D;
    // out is not read again by this operator, unless a fused projection reads it next
    const uint64_t pol_out = keep_out ? l2_evict_last() : l2_evict_first();

    for (int r0 = 0; r0 < nrows; r0 += BLK) {
        const int nb = min(BLK, nrows - r0);
        // ---- row sums ----
        bool ok = true;
        #pragma unroll
        for (int jr = 0; jr < BLK; ++jr) if (jr < nb) {
            const int i = r0 + jr;
            const int st = i % NST;
#ifdef ADALN_TEST_WAIT_NEVER_NS
            if (i == 0) ok = test_wait_never(&sm.never) && ok;
#endif
            ok = mbar_wait_bounded(&sm.full[wg][st], (uint32_t)(i / NST) & 1u) && ok;
            const unsigned char *row = my_stages + (size_t)st * row_bytes;
            float2 s1 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = t + 128 * j;
                if (v < V && ok) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(row + (size_t)v * 16);
                    s1 = f2add(s1, bf16x2_to_f2(w.x));
                    s1 = f2add(s1, bf16x2_to_f2(w.y));
                    s1 = f2add(s1, bf16x2_to_f2(w.z));
                    s1 = f2add(s1, bf16x2_to_f2(w.w));
                }
            }
            const float s1f = warp_sum(__fadd_rn(s1.x, s1.y));
            if (lane == 0) sm.red[wg][0][jr][warp] = s1f;
        }
        if (wg_barrier_or(1 + wg, !ok)) {
            if (t == 0) {
                report_error(kErrOutFwdWait);
                // let the copies this warp-group issued finish before leaving
                const int issued = min(nrows, r0 + NST);
                for (int k = r0; k < issued; ++k) drain_wait(&sm.full[wg][k % NST], (uint32_t)(k / NST) & 1u);
            }
            return;
        }
        if (t < nb) {
            float tot = sm.red[wg][0][t][0];
            tot = __fadd_rn(tot, sm.red[wg][0][t][1]);
            tot = __fadd_rn(tot, sm.red[wg][0][t][2]);
            tot = __fadd_rn(tot, sm.red[wg][0][t][3]);
            sm.mu[wg][t] = __fdiv_rn(tot, Df);
        }
        named_bar(1 + wg, 128);
        // ---- sums of squared deviations ----
        #pragma unroll
        for (int jr = 0; jr < BLK; ++jr) if (jr < nb) {
            const unsigned char *row = my_stages + (size_t)((r0 + jr) % NST) * row_bytes;
            const float2 mu2 = f2splat(sm.mu[wg][jr]);
            float2 s2 = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = t + 128 * j;
                if (v < V) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(row + (size_t)v * 16);
                    const uint32_t wa[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 c = f2sub(bf16x2_to_f2(wa[q]), mu2);
                        s2 = f2fma(c, c, s2);
                    }
                }
            }
            const float s2f = warp_sum(__fadd_rn(s2.x, s2.y));
            if (lane == 0) sm.red[wg][1][jr][warp] = s2f;
        }
        named_bar(1 + wg, 128);
        if (t < nb) {
            float tq = sm.red[wg][1][t][0];
            tq = __fadd_rn(tq, sm.red[wg][1][t][1]);
            tq = __fadd_rn(tq, sm.red[wg][1][t][2]);
            tq = __fadd_rn(tq, sm.red[wg][1][t][3]);
            sm.rs[wg][t] = __frsqrt_rn(__fadd_rn(__fdiv_rn(tq, Df), eps));
        }
        named_bar(1 + wg, 128);
        // ---- outputs ----
        #pragma unroll
        for (int jr = 0; jr < BLK; ++jr) if (jr < nb) {
            const int i = r0 + jr;
            const long long r = r_begin + i;
            const long long b = r / S;
            if (b != cur_b) {
                cur_b = b;
                const uint16_t *e = emb + (size_t)b * 2 * D;
#pragma unroll
                for (int j = 0; j < VPT; ++j) {
                    const int v = t + 128 * j;
                    if (v < V) {
                        const uint4 sc = ldg16(e + (size_t)v * 8);
                        const uint4 sh = ldg16(e + D + (size_t)v * 8);
                        const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};
                        const uint32_t shw[4] = {sh.x, sh.y, sh.z, sh.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float2 f = bf16x2_to_f2(scw[q]);
                            // onep = bf16(fp32(1 + scale))
                            onep[j][q] = make_float2(bf16f(bf16_bits(__fadd_rn(1.0f, f.x))),
                                                     bf16f(bf16_bits(__fadd_rn(1.0f, f.y))));
                            shift[j][q] = bf16x2_to_f2(shw[q]);
                        }
                    }
                }
            }
            const unsigned char *row = my_stages + (size_t)(i % NST) * row_bytes;
            const float mu = sm.mu[wg][jr], rs = sm.rs[wg][jr];
            const float2 mu2 = f2splat(mu), rs2 = f2splat(rs);
            uint16_t *orow = out + (size_t)r * D;
#pragma unroll
            for (int j = 0; j < VPT; ++j) {
                const int v = t + 128 * j;
                if (v < V) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(row + (size_t)v * 16);
                    const uint32_t wa[4] = {w.x, w.y, w.z, w.w};
                    uint32_t o[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float2 xh = f2mul(f2sub(bf16x2_to_f2(wa[q]), mu2), rs2);  // x_hat
                        // x_hat * onep is rounded before the shift is added (scalar: never fused)
                        const float2 pr = make_float2(__fmul_rn(xh.x, onep[j][q].x), __fmul_rn(xh.y, onep[j][q].y));
                        const float2 m = f2add(pr, shift[j][q]);
                        o[q] = pack_bf16x2(m.x, m.y);
                    }
                    stg16_hint(orow + (size_t)v * 8, make_uint4(o[0], o[1], o[2], o[3]), pol_out);
                }
            }
            if (t == 0) {
                mean[r] = mu;
                rstd[r] = rs;
            }
        }
        named_bar(1 + wg, 128);  // every thread is done with this block's stages
        if (t == 0)
            for (int jr = 0; jr < nb; ++jr) {
                const int i = r0 + jr;
                if (i + NST < nrows) {
                    const int st = i % NST;
                    mbar_arrive_expect_tx(&sm.full[wg][st], row_bytes);
                    bulk_g2s(my_stages + (size_t)st * row_bytes, x + (size_t)(r_begin + i + NST) * D, row_bytes,
                             &sm.full[wg][st]);
                }
            }
    }
}

// ==========================================================================
// Forward for rows of up to 8 KB (D <= 4096): one warp per token row, no
// barriers between warps.
//
// A CTA takes a range of rows of one sample b, and first puts the sample's
// onep = bf16(fp32(1 + scale)) and shift in shared memory as fp32.  Each warp
// takes the rows lo + w, lo + w + NW, ... of the range through a private ring
// of NS row buffers filled by 1-D bulk copies (the TMA engine); a row's 16-byte
// vectors v = lane + 32 j are copied into registers and the stage is handed
// back at once.  Row sums use shuffles only.  The reduction order over d: per
// lane, vectors j ascending into two packed accumulators (even j, odd j), the
// column pairs of a vector in order; the two accumulators, then the two halves
// of the pairs; then a fixed xor butterfly.  It depends on D only.
//
// RES (the block-level norm with a gated residual): a stage holds the x row and
// the residual row, the sample's gate sits in shared memory beside the table,
// and a lane forms r = bf16(residual + bf16(gate * x)) (eager bf16: each
// operation's fp32 result rounded once) for its vectors as it takes them from
// the stage, stores r, and normalises and modulates r as above.
// ==========================================================================
// EXACT: V == 32 * VPL, every lane's vectors lie inside the row (no tests)
template <int VPL, int MAXW, bool RES, bool EXACT>
__global__ void __launch_bounds__(MAXW * 32, 1)
out_fwd_row_kernel(const uint16_t *__restrict__ x, const uint16_t *__restrict__ emb, uint16_t *__restrict__ out,
                   float *__restrict__ mean, float *__restrict__ rstd, int S, int D, float eps, int cps, int NS,
                   int keep_out, const uint16_t *__restrict__ residual, const uint16_t *__restrict__ gate,
                   uint16_t *__restrict__ r_out) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int NW = blockDim.x >> 5;
    const int V = D >> 3;
    const int row_bytes = D * 2;
    // a stage holds the x row, and with RES the residual row after it
    const int stage_bytes = RES ? 2 * row_bytes : row_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_raw);             // [warps][NS] (+ 1: test builds)
    float *t_onep = reinterpret_cast<float *>(smem_raw + 1024);          // [D]
    float *t_shift = t_onep + D;                                         // [D]
    uint4 *t_gate = reinterpret_cast<uint4 *>(smem_raw + 1024 + (size_t)D * 8);  // RES: the sample's gate, [V]
    unsigned char *ring = smem_raw + 1024 + (size_t)D * (RES ? 10 : 8);  // [warps][NS][stage]
    unsigned char *my_ring = ring + (size_t)warp * NS * stage_bytes;
    uint64_t *my_full = full + warp * NS;

    const int b = blockIdx.x / cps;
    const int c = blockIdx.x % cps;
    const int lo = (int)(((long long)c * S) / cps);
    const int hi = (int)(((long long)(c + 1) * S) / cps);
    const int nrows = lo + warp < hi ? (hi - 1 - lo - warp) / NW + 1 : 0;  // rows of this warp
    const size_t row0 = (size_t)b * S + lo + warp;                        // first row; then + NW per row

    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&my_full[s], 1);
#ifdef ADALN_TEST_WAIT_NEVER_NS
        mbar_init(&full[MAXW * NS + warp], 1);  // this warp's never-completing barrier
#endif
        fence_barrier_init();
    }
    __syncwarp();
    pdl_wait();  // x and emb may come from preceding kernels
    // the sample's modulation parameters are requested before the row copies,
    // so that they do not queue behind them
    const uint16_t *e = emb + (size_t)b * 2 * D;
    uint4 sc0 = make_uint4(0u, 0u, 0u, 0u), sh0 = sc0;
    if ((int)threadIdx.x < V) {
        sc0 = ldg16(e + (size_t)threadIdx.x * 8);
        sh0 = ldg16(e + D + (size_t)threadIdx.x * 8);
    }
    if (lane == 0)
        for (int k = 0; k < NS && k < nrows; ++k) {
            unsigned char *dst = my_ring + (size_t)k * stage_bytes;
            mbar_arrive_expect_tx(&my_full[k], stage_bytes);
            bulk_g2s(dst, x + (row0 + (size_t)k * NW) * D, row_bytes, &my_full[k]);
            if (RES) bulk_g2s(dst + row_bytes, residual + (row0 + (size_t)k * NW) * D, row_bytes, &my_full[k]);
        }
    if (RES)
        for (int i = threadIdx.x; i < V; i += blockDim.x) t_gate[i] = ldg16(gate + (size_t)b * D + (size_t)i * 8);
    // the sample's modulation parameters, fp32
    for (int i = threadIdx.x; i < V; i += blockDim.x) {
        const uint4 sc = i == (int)threadIdx.x ? sc0 : ldg16(e + (size_t)i * 8);
        const uint4 sh = i == (int)threadIdx.x ? sh0 : ldg16(e + D + (size_t)i * 8);
        const uint32_t scw[4] = {sc.x, sc.y, sc.z, sc.w};
        const uint32_t shw[4] = {sh.x, sh.y, sh.z, sh.w};
        float on[8], sf[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            on[2 * q] = bf16f(bf16_bits(__fadd_rn(1.0f, bf16lo(scw[q]))));
            on[2 * q + 1] = bf16f(bf16_bits(__fadd_rn(1.0f, bf16hi(scw[q]))));
            sf[2 * q] = bf16lo(shw[q]);
            sf[2 * q + 1] = bf16hi(shw[q]);
        }
        // two planes of float4 (columns 0-3, then 4-7 of every vector), so that
        // the lanes of a warp read consecutive 16-byte words
        float4 *po = reinterpret_cast<float4 *>(t_onep);
        float4 *ps = reinterpret_cast<float4 *>(t_shift);
        po[i] = make_float4(on[0], on[1], on[2], on[3]);
        po[V + i] = make_float4(on[4], on[5], on[6], on[7]);
        ps[i] = make_float4(sf[0], sf[1], sf[2], sf[3]);
        ps[V + i] = make_float4(sf[4], sf[5], sf[6], sf[7]);
    }
    __syncthreads();
    pdl_trigger();

    const float Df = (float)D;
    // out is not read again by this operator, unless a fused projection reads it next
    const uint64_t pol_out = keep_out ? l2_evict_last() : l2_evict_first();
    const uint64_t pol_r = l2_evict_first();
    for (int k = 0; k < nrows; ++k) {
        const size_t r = row0 + (size_t)k * NW;
        const int st = k % NS;
#ifdef ADALN_TEST_WAIT_NEVER_NS
        const bool ok = (k == 0 ? test_wait_never(&full[MAXW * NS + warp]) : true) &&
                        mbar_wait_bounded(&my_full[st], (uint32_t)(k / NS) & 1u);
#else
        const bool ok = mbar_wait_bounded(&my_full[st], (uint32_t)(k / NS) & 1u);
#endif
        if (__any_sync(0xFFFFFFFFu, !ok)) {
            if (lane == 0) {
                report_error(kErrOutFwdWait);
                // let the copies this warp issued finish before leaving
                const int issued = min(nrows, k + NS);
                for (int q = k; q < issued; ++q) drain_wait(&my_full[q % NS], (uint32_t)(q / NS) & 1u);
            }
            return;
        }
        const uint4 *srow = reinterpret_cast<const uint4 *>(my_ring + (size_t)st * stage_bytes);
        uint4 xr[VPL];
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int v = lane + 32 * j;
            xr[j] = (EXACT || v < V) ? srow[v] : make_uint4(0u, 0u, 0u, 0u);
            if (RES && (EXACT || v < V)) {
                // the gated residual, in eager bf16: r = bf16(residual + bf16(gate * x)); r is normalised below
                const uint4 rv = srow[V + v], gv = t_gate[v];
                const uint32_t xa[4] = {xr[j].x, xr[j].y, xr[j].z, xr[j].w}, ra[4] = {rv.x, rv.y, rv.z, rv.w},
                               ga[4] = {gv.x, gv.y, gv.z, gv.w};
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    o[q] = pack_bf16x2(eager_add(bf16lo(ra[q]), eager_mul(bf16lo(ga[q]), bf16lo(xa[q]))),
                                       eager_add(bf16hi(ra[q]), eager_mul(bf16hi(ga[q]), bf16hi(xa[q]))));
                xr[j] = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        __syncwarp();  // every lane has its part of the row: refill the stage
        if (lane == 0 && k + NS < nrows) {
            unsigned char *dst = my_ring + (size_t)st * stage_bytes;
            mbar_arrive_expect_tx(&my_full[st], stage_bytes);
            bulk_g2s(dst, x + (r + (size_t)NS * NW) * D, row_bytes, &my_full[st]);
            if (RES) bulk_g2s(dst + row_bytes, residual + (r + (size_t)NS * NW) * D, row_bytes, &my_full[st]);
        }
        if (RES) {
            // r is read again only by the backward: streamed out
            uint16_t *rrow = r_out + r * D;
#pragma unroll
            for (int j = 0; j < VPL; ++j) {
                const int v = lane + 32 * j;
                if (EXACT || v < V) stg16_hint(rrow + (size_t)v * 8, xr[j], pol_r);
            }
        }
        // mean (zero vectors past the row end add +0 and change nothing)
        float2 s1[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            s1[j & 1] = f2add(s1[j & 1], bf16x2_to_f2(xr[j].x));
            s1[j & 1] = f2add(s1[j & 1], bf16x2_to_f2(xr[j].y));
            s1[j & 1] = f2add(s1[j & 1], bf16x2_to_f2(xr[j].z));
            s1[j & 1] = f2add(s1[j & 1], bf16x2_to_f2(xr[j].w));
        }
        const float2 t1 = f2add(s1[0], s1[1]);
        const float mu = __fdiv_rn(warp_sum(__fadd_rn(t1.x, t1.y)), Df);
        const float2 mu2 = f2splat(mu);
        // variance
        float2 s2[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            if (EXACT || lane + 32 * j < V) {
                const uint32_t wa[4] = {xr[j].x, xr[j].y, xr[j].z, xr[j].w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 d = f2sub(bf16x2_to_f2(wa[q]), mu2);
                    s2[j & 1] = f2fma(d, d, s2[j & 1]);
                }
            }
        }
        const float2 t2 = f2add(s2[0], s2[1]);
        const float var = __fdiv_rn(warp_sum(__fadd_rn(t2.x, t2.y)), Df);
        const float rs = __frsqrt_rn(__fadd_rn(var, eps));
        const float2 rs2 = f2splat(rs);
        // outputs
        uint16_t *orow = out + r * D;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int v = lane + 32 * j;
            if (EXACT || v < V) {
                const float4 *po = reinterpret_cast<const float4 *>(t_onep);
                const float4 *ps = reinterpret_cast<const float4 *>(t_shift);
                const float4 oa = po[v], ob = po[V + v], sa = ps[v], sb = ps[V + v];
                const float2 onp[4] = {make_float2(oa.x, oa.y), make_float2(oa.z, oa.w), make_float2(ob.x, ob.y),
                                       make_float2(ob.z, ob.w)};
                const float2 shf[4] = {make_float2(sa.x, sa.y), make_float2(sa.z, sa.w), make_float2(sb.x, sb.y),
                                       make_float2(sb.z, sb.w)};
                const uint32_t wa[4] = {xr[j].x, xr[j].y, xr[j].z, xr[j].w};
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float2 xh = f2mul(f2sub(bf16x2_to_f2(wa[q]), mu2), rs2);  // x_hat
                    // x_hat * onep is rounded before the shift is added (scalar: never fused)
                    const float2 pr = make_float2(__fmul_rn(xh.x, onp[q].x), __fmul_rn(xh.y, onp[q].y));
                    const float2 m = f2add(pr, shf[q]);
                    o[q] = pack_bf16x2(m.x, m.y);
                }
                stg16_hint(orow + (size_t)v * 8, make_uint4(o[0], o[1], o[2], o[3]), pol_out);
            }
        }
        if (lane == 0) {
            mean[r] = mu;
            rstd[r] = rs;
        }
    }
}

template <int VPL, int MAXW, bool RES = false>
static cudaError_t launch_out_fwd_row(const uint16_t *x, const uint16_t *emb, uint16_t *out, float *mean,
                                      float *rstd, int B, int S, int D, float eps, cudaStream_t stream,
                                      const DeviceInfo &dev, bool keep_out, const uint16_t *residual = nullptr,
                                      const uint16_t *gate = nullptr, uint16_t *r_out = nullptr) {
    constexpr size_t kSmemMax = 227 * 1024;
    const size_t stage = (size_t)D * 2 * (RES ? 2 : 1);
    auto smem_of = [&](int warps, int ns) { return 1024 + (size_t)D * (RES ? 10 : 8) + (size_t)warps * ns * stage; };
    int warps, ns;
    if (!RES) {
        // 16 warps with 2 stages each where that fits, else 8 warps with 3 (or 2)
        warps = 8;
        ns = smem_of(8, 3) <= kSmemMax ? 3 : 2;
        if (MAXW == 16 && smem_of(16, 2) <= kSmemMax) { warps = 16; ns = 2; }
    } else {
        // two rows per stage: all the warps with 2 stages, else with 1
        warps = MAXW;
        ns = smem_of(MAXW, 2) <= kSmemMax ? 2 : 1;
        if (smem_of(warps, ns) > kSmemMax) warps = 8;
    }
    const size_t smem = smem_of(warps, ns);
    auto kern = D / 8 == 32 * VPL ? out_fwd_row_kernel<VPL, MAXW, RES, true> : out_fwd_row_kernel<VPL, MAXW, RES, false>;
    cudaError_t err = ensure_smem_attr((const void *)kern, smem, dev);
    if (err != cudaSuccess) return err;
    // about one CTA per SM in all; every CTA within one sample
    int cps = (dev.sm_count + B - 1) / B;
    if (cps > S) cps = S;
    if (cps < 1) cps = 1;
    const long long grid = (long long)B * cps;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(warps * 32), smem, stream, x, emb, out, mean, rstd, S, D, eps,
                      cps, ns, keep_out ? 1 : 0, residual, gate, r_out);
}

template <int VPT, int BLK, int NST, int MINB>
static cudaError_t launch_out_fwd_t(const uint16_t *x, const uint16_t *emb, uint16_t *out, float *mean,
                                    float *rstd, int B, int S, int D, float eps, cudaStream_t stream,
                                    const DeviceInfo &dev, bool keep_out) {
    static_assert(NST == 2 * BLK && BLK <= kFwdBlock, "two blocks of rows in flight");
    const size_t smem = ((sizeof(FwdSmem) + 127) / 128) * 128 + (size_t)kWG * NST * D * 2;
    auto kern = out_fwd_kernel<VPT, BLK, NST, MINB>;
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
                      x, emb, out, mean, rstd, S, D, eps, R, keep_out ? 1 : 0);
}

// Rows of up to 8 KB (D <= 4096): one warp per row.  Longer rows: the
// warp-group kernel, with blocks of 2 rows and 4 stages (128 KB of stages).
cudaError_t launch_out_fwd(const uint16_t *x, const uint16_t *emb, uint16_t *out, float *mean, float *rstd,
                           int B, int S, int D, float eps, cudaStream_t stream, const DeviceInfo &dev, bool keep_out) {
    const int V = D / 8;
    if (V <= 128) return launch_out_fwd_row<4, 16>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, keep_out);
    if (V <= 256) return launch_out_fwd_row<8, 16>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, keep_out);
    if (V <= 384) return launch_out_fwd_row<12, 16>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, keep_out);
    if (V <= 512) return launch_out_fwd_row<16, 8>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, keep_out);
    const int vpt = (V + 127) / 128;
    switch (vpt) {
        case 1: return launch_out_fwd_t<1, 4, 8, 2>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, keep_out);
        case 2: return launch_out_fwd_t<2, 4, 8, 2>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, keep_out);
        case 3: return launch_out_fwd_t<3, 4, 8, 2>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, keep_out);
        case 4: return launch_out_fwd_t<4, 4, 8, 1>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, keep_out);
        case 5: case 6: return launch_out_fwd_t<6, 2, 4, 1>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, keep_out);
        default: return launch_out_fwd_t<8, 2, 4, 1>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, keep_out);
    }
}

// The block-level norm's forward in one kernel (rows of up to 8 KB): r =
// bf16(residual + bf16(gate * x)) is formed from staged x and residual rows,
// written, and normalised and modulated in registers, so r is never read back.
bool out_fwd_res_supported(int D) { return D / 8 <= 512; }

cudaError_t launch_out_fwd_res(const uint16_t *x, const uint16_t *residual, const uint16_t *gate,
                               const uint16_t *emb, uint16_t *r, uint16_t *out, float *mean, float *rstd, int B,
                               int S, int D, float eps, cudaStream_t stream, const DeviceInfo &dev) {
    const int V = D / 8;
    if (V <= 128)
        return launch_out_fwd_row<4, 16, true>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, false, residual,
                                               gate, r);
    if (V <= 256)
        return launch_out_fwd_row<8, 16, true>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, false, residual,
                                               gate, r);
    if (V <= 384)
        return launch_out_fwd_row<12, 16, true>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, false, residual,
                                                gate, r);
    return launch_out_fwd_row<16, 8, true>(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, false, residual, gate,
                                           r);
}

// ==========================================================================
// Backward, kernel 1: one CTA per (sample b, 32-token tile t).
//
// Thread i owns the 16-byte vectors v = i + NT j (8 columns each); all its
// fp32 arithmetic is packed (column pairs), in inline PTX with explicit
// rounding, so no product is ever fused into the add that consumes it.  Rows
// arrive through a ring of NST stages (an x row and a dy row each) filled by
// bulk copies, and are taken in blocks of RB rows.
//
// Phase 1, per row in ascending s: x_hat = (x - mean) * rstd (bit-identical to
// the forward's value), g = fp32(dy), the token product p = g * x_hat (rounded);
// p and g go into the columns' level-0 tree nodes by TwoSum (the Neumaier step,
// branch-free), and each thread keeps partial row sums of g * onep and
// p * onep.  The warp reduces the block's sums at once (column pairs' halves,
// then a fixed transposed butterfly) and publishes them; after one CTA barrier
// every warp adds the warps' sums in ascending order (every warp the same
// bits): c1 = sum_d g onep / D, c2 = sum_d g x_hat onep / D.  Phase 2 writes
//     dx = rstd gh + (mean rstd^2 c2 - rstd c1) - x rstd^2 c2,   gh = g * onep,
// which is rstd (gh - c1 - x_hat c2), two fused multiply-adds per column pair
// after one multiply.  The reduction order over d depends on D only.  A block's
// stages are refilled by the last warp to finish its phase 2 (a counter per
// block of stages), while the other warps go on.
// ==========================================================================
constexpr int kRowBlock = 4;        // most rows per block
constexpr int kBwdMaxStages = 8;

struct BwdSmem {
    float2 red[2][kRowBlock][32];   // [block parity][row of the block][warp] = (sum g onep, sum p onep)
    float mu[kTile], rs[kTile];
    uint64_t full[kBwdMaxStages];   // a stage's copies have landed
    unsigned rel[kBwdMaxStages];    // warps done with the rows of a block of stages
    int last[kBwdMaxStages];        // latest row copied into a stage (-1: none)
    int abort;                      // a wait ran out of time
    ADALN_NEVER_BAR
};

// The NV partial sums of a warp's lanes reduced at once (a transposed
// butterfly): at the first log2(NV) levels a lane keeps half of its values and
// adds the partner's copy of them, then plain levels follow; lane l ends with
// value l >> (5 - log2 NV) summed over all 32 lanes, in a fixed tree.
template <int NV>
__device__ __forceinline__ float warp_transposed_sum(const float (&in)[NV], int lane) {
    static_assert(NV == 2 || NV == 4 || NV == 8, "2, 4 or 8 values");
    float a[NV];
#pragma unroll
    for (int q = 0; q < NV; ++q) a[q] = in[q];
#pragma unroll
    for (int off = 16, cnt = NV; off >= 1; off >>= 1) {
        if (cnt > 1) {
            const bool up = (lane & off) != 0;
#pragma unroll
            for (int q = 0; q < NV / 2; ++q) {
                if (q < cnt / 2) {
                    const float keep = up ? a[q + cnt / 2] : a[q];
                    const float give = up ? a[q] : a[q + cnt / 2];
                    a[q] = __fadd_rn(keep, __shfl_xor_sync(0xFFFFFFFFu, give, off));
                }
            }
            cnt /= 2;
        } else {
            a[0] = __fadd_rn(a[0], __shfl_xor_sync(0xFFFFFFFFu, a[0], off));
        }
    }
    return a[0];
}

template <int VPT, int MAXNT, int MINB, int RB, int NST, bool EXACT>
__global__ void __launch_bounds__(MAXNT, MINB)
out_bwd_tile_kernel(const uint16_t *__restrict__ dy, const uint16_t *__restrict__ x,
                    const uint16_t *__restrict__ emb, const float *__restrict__ mean,
                    const float *__restrict__ rstd, uint16_t *__restrict__ dx, float *__restrict__ ws_sig,
                    float *__restrict__ ws_kap, int S, int D, int T, int keep_dx) {
    static_assert((RB == 1 || RB == 2 || RB == 4) && NST >= 2 * RB && NST <= kBwdMaxStages && NST % RB == 0,
                  "whole blocks of rows per stage group, two blocks in flight");
    extern __shared__ __align__(128) unsigned char smem_raw[];
    BwdSmem &sm = *reinterpret_cast<BwdSmem *>(smem_raw);
    volatile int *abort_flag = &sm.abort;
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
        for (int s = 0; s < NST; ++s) {
            mbar_init(&sm.full[s], 1);
            sm.rel[s] = 0u;
            sm.last[s] = -1;
        }
        sm.abort = 0;
#ifdef ADALN_TEST_WAIT_NEVER_NS
        mbar_init(&sm.never, 1);
#endif
        fence_barrier_init();
    }
    __syncthreads();
    pdl_wait();  // mean, rstd, emb (and perhaps x, dy) come from preceding kernels
    pdl_trigger();

    // the row statistics and the sample's scale are requested before the row
    // copies, so that they do not queue behind them
    float mu_t = 0.0f, rs_t = 0.0f;
    if (tid < n) {
        mu_t = mean[row0 + tid];
        rs_t = rstd[row0 + tid];
    }
    const uint16_t *e = emb + (size_t)b * 2 * D;
    uint4 sc_v[VPT];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tid + NT * j;
        sc_v[j] = (EXACT || v < V) ? ldg16(e + (size_t)v * 8) : make_uint4(0u, 0u, 0u, 0u);
    }
    // dy and dx are streamed once: evict-first in L2 (dx evict-last when a
    // following kernel of the same call reads it)
    const uint64_t pol_stream = l2_evict_first();
    const uint64_t pol_dx = keep_dx ? l2_evict_last() : pol_stream;
    if (tid == 0) {
        for (int i = 0; i < NST && i < n; ++i) {
            unsigned char *dst = stages + (size_t)i * stage_bytes;
            mbar_arrive_expect_tx(&sm.full[i], stage_bytes);
            bulk_g2s(dst, x + (row0 + i) * D, row_bytes, &sm.full[i]);
            bulk_g2s_hint(dst + row_bytes, dy + (row0 + i) * D, row_bytes, &sm.full[i], pol_stream);
            sm.last[i] = i;
        }
    }
    if (tid < n) {
        sm.mu[tid] = mu_t;
        sm.rs[tid] = rs_t;
    }
    // onep = bf16(fp32(1 + scale)) of this thread's columns, by column pair
    px2 onep[VPT][4];
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const uint32_t w[4] = {sc_v[j].x, sc_v[j].y, sc_v[j].z, sc_v[j].w};
#pragma unroll
        for (int q = 0; q < 4; ++q)
            onep[j][q] = px_make(bf16f(bf16_bits(__fadd_rn(1.0f, bf16lo(w[q])))),
                                 bf16f(bf16_bits(__fadd_rn(1.0f, bf16hi(w[q])))));
    }
    __syncthreads();

    // Tree nodes of the scale products p = g * x_hat and of the shift products
    // g, by column pair.  They start at +0 rather than at the first token:
    // adding a value v to +0 gives v exactly with no error, so every later step
    // is the same; only an all-zero column can differ, in the sign of its
    // level-0 sum (+0 for -0), and its root (sum + correction) is +0 either way.
    px2 sg_s[VPT][4], kp_s[VPT][4], sg_h[VPT][4], kp_h[VPT][4];
#pragma unroll
    for (int j = 0; j < VPT; ++j)
#pragma unroll
        for (int q = 0; q < 4; ++q) sg_s[j][q] = kp_s[j][q] = sg_h[j][q] = kp_h[j][q] = 0ull;
    const float invD = __frcp_rn((float)D);  // c1, c2 only feed dx (tolerance-checked)

    // phase 1 of one row, its sums into rsum[2 jr], rsum[2 jr + 1]; EXACT: every
    // thread's vectors lie inside the row (no bounds test, so the tree state
    // stays in the same registers on every path)
    auto phase1_row = [&](int i, int jr, float (&rsum)[2 * RB]) {
        const unsigned char *xs = stages + (size_t)(i % NST) * stage_bytes;
        const unsigned char *gs = xs + row_bytes;
        const px2 mu2 = px_splat(sm.mu[i]), rs2 = px_splat(sm.rs[i]);
        px2 a1 = 0ull, a2 = 0ull;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = tid + NT * j;
            if (EXACT || v < V) {
                const uint4 xw = *reinterpret_cast<const uint4 *>(xs + (size_t)v * 16);
                const uint4 gw = *reinterpret_cast<const uint4 *>(gs + (size_t)v * 16);
                const uint32_t xa[4] = {xw.x, xw.y, xw.z, xw.w};
                const uint32_t ga[4] = {gw.x, gw.y, gw.z, gw.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const px2 g2 = px_bf16(ga[q]);
                    const px2 xh = px_mul(px_sub(px_bf16(xa[q]), mu2), rs2);  // x_hat
                    const px2 p = px_mul(g2, xh);  // rounded before it enters the tree
                    a1 = px_fma(g2, onep[j][q], a1);
                    a2 = px_fma(p, onep[j][q], a2);
                    px_twosum(sg_s[j][q], kp_s[j][q], p);
                    px_twosum(sg_h[j][q], kp_h[j][q], g2);
                }
            }
        }
        rsum[2 * jr] = __fadd_rn(px_lo(a1), px_hi(a1));
        rsum[2 * jr + 1] = __fadd_rn(px_lo(a2), px_hi(a2));
    };
    // phase 2 of one row: dx from the row's constants k2 = rstd^2 c2 and
    // k3 = mean k2 - rstd c1
    auto phase2_row = [&](int i, float k2, float k3) {
        const unsigned char *xs = stages + (size_t)(i % NST) * stage_bytes;
        const unsigned char *gs = xs + row_bytes;
        const px2 rs2 = px_splat(sm.rs[i]), nk2 = px_splat(-k2), k3v = px_splat(k3);
        uint16_t *drow = dx + (row0 + i) * D;
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = tid + NT * j;
            if (EXACT || v < V) {
                const uint4 xw = *reinterpret_cast<const uint4 *>(xs + (size_t)v * 16);
                const uint4 gw = *reinterpret_cast<const uint4 *>(gs + (size_t)v * 16);
                const uint32_t xa[4] = {xw.x, xw.y, xw.z, xw.w};
                const uint32_t ga[4] = {gw.x, gw.y, gw.z, gw.w};
                uint32_t o[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const px2 gh = px_mul(px_bf16(ga[q]), onep[j][q]);
                    const px2 t = px_fma(px_bf16(xa[q]), nk2, k3v);
                    o[q] = px_to_bf16x2(px_fma(gh, rs2, t));
                }
                stg16_hint(drow + (size_t)v * 8, make_uint4(o[0], o[1], o[2], o[3]), pol_dx);
            }
        }
    };

    const int nblk = (n + RB - 1) / RB;
    bool ok = true;
    for (int blk = 0; blk < nblk; ++blk) {
        const int r0 = blk * RB;
        const int nb = min(RB, n - r0);
        // ---- phase 1: tree products and the row sums ----
        bool landed = true;
#ifdef ADALN_TEST_WAIT_NEVER_NS
        if (blk == 0) landed = test_wait_never(&sm.never);
#endif
#pragma unroll
        for (int jr = 0; jr < RB; ++jr)
            if (jr < nb)
                landed = mbar_wait_or_abort(&sm.full[(r0 + jr) % NST], (uint32_t)((r0 + jr) / NST) & 1u,
                                            abort_flag) && landed;
        landed = __all_sync(0xFFFFFFFFu, landed);
        float rsum[2 * RB];  // this thread's (sum g onep, sum p onep) of each row of the block
#pragma unroll
        for (int q = 0; q < 2 * RB; ++q) rsum[q] = 0.0f;
        if (landed) {
            if (nb == RB) {
#pragma unroll
                for (int jr = 0; jr < RB; ++jr) phase1_row(r0 + jr, jr, rsum);
            } else {  // the short last block of a ragged tile
#pragma unroll
                for (int jr = 0; jr < RB; ++jr)
                    if (jr < nb) phase1_row(r0 + jr, jr, rsum);
            }
        }
        // publish the warp's sums of the block: lane l holds value l >> (5 - log2(2 RB))
        {
            const float v = warp_transposed_sum<2 * RB>(rsum, lane);
            constexpr int kShift = RB == 4 ? 2 : (RB == 2 ? 3 : 4);
            const int idx = lane >> kShift;
            if ((lane & ((1 << kShift) - 1)) == 0) {
                float *dst = reinterpret_cast<float *>(&sm.red[blk & 1][idx >> 1][warp]);
                dst[idx & 1] = v;
            }
        }
        if (__syncthreads_or(!landed)) {
            ok = false;
            break;
        }
        // ---- phase 2: dx ----
        // lane l < 2 nb: quantity (l & 1) of row (l >> 1), the warps added in ascending order
        float cs = 0.0f;
        if (lane < 2 * nb) {
            const float *src = reinterpret_cast<const float *>(&sm.red[blk & 1][lane >> 1][0]) + (lane & 1);
            cs = src[0];
            for (int w = 1; w < nwarps; ++w) cs = __fadd_rn(cs, src[2 * w]);
            cs = __fmul_rn(cs, invD);
        }
        // dx = rstd (gh - c1 - x_hat c2) = rstd gh + (mean k2 - rstd c1) - x k2,  k2 = rstd^2 c2
        const float c2 = __shfl_down_sync(0xFFFFFFFFu, cs, 1);
        float k2 = 0.0f, k3 = 0.0f;
        if ((lane & 1) == 0 && lane < 2 * nb) {
            const float rsv = sm.rs[r0 + (lane >> 1)], muv = sm.mu[r0 + (lane >> 1)];
            k2 = __fmul_rn(__fmul_rn(rsv, rsv), c2);
            k3 = __fmaf_rn(muv, k2, -__fmul_rn(rsv, cs));
        }
        if (nb == RB) {
#pragma unroll
            for (int jr = 0; jr < RB; ++jr)
                phase2_row(r0 + jr, __shfl_sync(0xFFFFFFFFu, k2, 2 * jr), __shfl_sync(0xFFFFFFFFu, k3, 2 * jr));
        } else {
#pragma unroll
            for (int jr = 0; jr < RB; ++jr) {
                const float kk2 = __shfl_sync(0xFFFFFFFFu, k2, 2 * jr), kk3 = __shfl_sync(0xFFFFFFFFu, k3, 2 * jr);
                if (jr < nb) phase2_row(r0 + jr, kk2, kk3);
            }
        }
        // this warp is done with the block's stages; the last warp to finish
        // refills them with the rows NST further on
        __syncwarp();
        if (lane == 0) {
            const int grp = blk % (NST / RB);
            if (smem_add_acq_rel(&sm.rel[grp], 1u) == (unsigned)nwarps - 1u) {
                sm.rel[grp] = 0u;
                fence_proxy_async_smem();
                for (int jr = 0; jr < nb; ++jr) {
                    const int i = r0 + jr;
                    const int st = i % NST;
                    if (i + NST < n) {
                        unsigned char *dst = stages + (size_t)st * stage_bytes;
                        mbar_arrive_expect_tx(&sm.full[st], stage_bytes);
                        bulk_g2s(dst, x + (row0 + i + NST) * D, row_bytes, &sm.full[st]);
                        bulk_g2s_hint(dst + row_bytes, dy + (row0 + i + NST) * D, row_bytes, &sm.full[st],
                                      pol_stream);
                        sm.last[st] = i + NST;
                    }
                }
            }
        }
    }
    if (!ok) {
        // every thread left the loop at the same barrier: no copy is issued any more
        if (tid == 0) {
            report_error(kErrOutBwdWait);
            // let the copies this CTA issued land before it leaves
            for (int st = 0; st < NST; ++st)
                if (sm.last[st] >= 0) drain_wait(&sm.full[st], (uint32_t)(sm.last[st] / NST) & 1u);
        }
        return;
    }
    // level-0 node of this tile: scale half at columns [0, D), shift half at [D, 2D);
    // kept in L2 (evict-last) for the fold that reads it next
    const int H = 2 * D;
    float *ps = ws_sig + ((size_t)b * T + tile) * H;
    float *pk = ws_kap + ((size_t)b * T + tile) * H;
    const uint64_t pol_keep = l2_evict_last();
    auto put = [&](float *dst, px2 a, px2 c) {
        stg16f_hint(dst, make_float4(px_lo(a), px_hi(a), px_lo(c), px_hi(c)), pol_keep);
    };
#pragma unroll
    for (int j = 0; j < VPT; ++j) {
        const int v = tid + NT * j;
        if (EXACT || v < V) {
            const size_t c = (size_t)v * 8;
            put(ps + c, sg_s[j][0], sg_s[j][1]);
            put(ps + c + 4, sg_s[j][2], sg_s[j][3]);
            put(pk + c, kp_s[j][0], kp_s[j][1]);
            put(pk + c + 4, kp_s[j][2], kp_s[j][3]);
            put(ps + D + c, sg_h[j][0], sg_h[j][1]);
            put(ps + D + c + 4, sg_h[j][2], sg_h[j][3]);
            put(pk + D + c, kp_h[j][0], kp_h[j][1]);
            put(pk + D + c + 4, kp_h[j][2], kp_h[j][3]);
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
// lane = column.  Warp w folds the level-1 groups w, w + W, ... straight from
// the level-0 nodes in global memory, all 32 children of a group requested at
// once (one round trip); higher levels fold in shared memory.
// ==========================================================================
// shared memory of the fold: level-1 nodes s1, k1 [n1][32], then level-2
// nodes s2, k2 [ceil(n1/32)][32] (n1 = ceil(T/32) <= 256)
__host__ __device__ constexpr size_t fold_smem_bytes(int n1) {
    return n1 <= 1 ? 0 : (size_t)2 * 32 * sizeof(float) * (n1 + (n1 + kTile - 1) / kTile);
}

// One group: Neumaier sum of the children's sums in ascending order
// (compensation c), the children's corrections added in ascending order;
// node = (sum, c + corrections).
__device__ __forceinline__ void fold_values(const float (&vs)[kTile], const float (&vk)[kTile], int count,
                                            float &out_s, float &out_k) {
    float s = vs[0], k = vk[0], c = 0.0f;
#pragma unroll
    for (int q = 1; q < kTile; ++q) {
        if (q < count) {
            twosum(s, c, vs[q]);
            k = __fadd_rn(k, vk[q]);
        }
    }
    out_s = s;
    out_k = __fadd_rn(c, k);
}

__device__ __forceinline__ void fold_group(const float *sig, const float *kap, size_t stride, int count,
                                           float &out_s, float &out_k) {
    float vs[kTile], vk[kTile];
    const uint64_t pol = l2_evict_first();  // the level-0 nodes are read once
    if (count == kTile) {
        // a full group: all 64 loads issued before the first add
#pragma unroll
        for (int q = 0; q < kTile; ++q) vs[q] = ldcg_hint(sig + (size_t)q * stride, pol);
#pragma unroll
        for (int q = 0; q < kTile; ++q) vk[q] = ldcg_hint(kap + (size_t)q * stride, pol);
    } else {
#pragma unroll
        for (int q = 0; q < kTile; ++q) {
            vs[q] = q < count ? ldcg_hint(sig + (size_t)q * stride, pol) : 0.0f;
            vk[q] = q < count ? ldcg_hint(kap + (size_t)q * stride, pol) : 0.0f;
        }
    }
    fold_values(vs, vk, count, out_s, out_k);
}

// the same over shared memory (levels >= 2)
__device__ __forceinline__ void fold_group_smem(const float *sig, const float *kap, int count, float &out_s,
                                                float &out_k) {
    float vs[kTile], vk[kTile];
#pragma unroll
    for (int q = 0; q < kTile; ++q) {
        vs[q] = q < count ? sig[q * 32] : 0.0f;
        vk[q] = q < count ? kap[q * 32] : 0.0f;
    }
    fold_values(vs, vk, count, out_s, out_k);
}

constexpr int kFoldWarps = 8;

__global__ void __launch_bounds__(kFoldWarps * 32)
tree_fold_kernel(const float *__restrict__ ws_sig, const float *__restrict__ ws_kap, float *__restrict__ out,
                 int T, int H) {
    extern __shared__ __align__(128) float fold_sh[];
    pdl_wait();
    pdl_trigger();  // the next kernel may become resident and wait; it reads out only after its own wait
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int W = blockDim.x >> 5;
    const int b = blockIdx.y;
    const int col = blockIdx.x * 32 + lane;
    const bool live = col < H;
    const size_t base = (size_t)b * T * H + (size_t)(live ? col : 0);

    if (T == 1) {  // the tile is the root
        if (warp == 0 && live) out[(size_t)b * H + col] = __fadd_rn(ws_sig[base], ws_kap[base]);
        return;
    }
    const int n1 = (T + kTile - 1) / kTile;
    const int m2 = (n1 + kTile - 1) / kTile;
    float(*s1)[32] = reinterpret_cast<float(*)[32]>(fold_sh);
    float(*k1)[32] = s1 + n1;
    float(*s2)[32] = k1 + n1;
    float(*k2)[32] = s2 + m2;
    for (int gi = warp; gi < n1; gi += W) {
        const int i0 = gi * kTile;
        const int cnt = min(kTile, T - i0);
        float s, k;
        fold_group(ws_sig + base + (size_t)i0 * H, ws_kap + base + (size_t)i0 * H, (size_t)H, cnt, s, k);
        if (n1 == 1) {  // the level-1 node is the root
            if (live) out[(size_t)b * H + col] = __fadd_rn(s, k);
            return;
        }
        s1[gi][lane] = s;
        k1[gi][lane] = k;
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
                fold_group_smem(&s1[i0][lane], &k1[i0][lane], cnt, s, k);
                s2[gi][lane] = s;
                k2[gi][lane] = k;
            } else {
                fold_group_smem(&s2[i0][lane], &k2[i0][lane], cnt, s, k);
                s1[gi][lane] = s;
                k1[gi][lane] = k;
            }
        }
        __syncthreads();
        in_first = !in_first;
        nn = m;
    }
    if (warp == 0 && live) {
        const float s = in_first ? s1[0][lane] : s2[0][lane];
        const float k = in_first ? k1[0][lane] : k2[0][lane];
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
cudaError_t launch_fold(const float *sig, const float *kap, float *out, int B, int T, int H, cudaStream_t stream,
                        const DeviceInfo &dev) {
    const int n1 = (T + kTile - 1) / kTile;
    const int warps = T == 1 ? 1 : min(kFoldWarps, n1);
    const size_t smem = fold_smem_bytes(n1);
    cudaError_t err = ensure_smem_attr((const void *)tree_fold_kernel, smem, dev);
    if (err != cudaSuccess) return err;
    return launch_pdl(tree_fold_kernel, dim3((H + 31) / 32, B), dim3(32 * warps), smem, stream,
                      sig, kap, out, T, H);
}

cudaError_t launch_zero(float *p, size_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    return launch_pdl(zero_kernel, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, stream, p, n);
}

template <int VPT, int MAXNT, int MINB, int RB, int NST>
static cudaError_t launch_out_bwd_t(const uint16_t *dy, const uint16_t *x, const uint16_t *emb, const float *mean,
                                    const float *rstd, uint16_t *dx, float *sig, float *kap, int B, int S, int D,
                                    int T, cudaStream_t stream, const DeviceInfo &dev, bool keep_dx) {
    const int V = D / 8;
    const int nt = ((V + VPT - 1) / VPT + 31) / 32 * 32;
    const size_t smem = ((sizeof(BwdSmem) + 127) / 128) * 128 + (size_t)NST * 4 * D;
    // every thread's vectors inside the row: the form without bounds tests
    auto kern = nt * VPT == V ? out_bwd_tile_kernel<VPT, MAXNT, MINB, RB, NST, true>
                              : out_bwd_tile_kernel<VPT, MAXNT, MINB, RB, NST, false>;
    cudaError_t err = ensure_smem_attr((const void *)kern, smem, dev);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(T, B), dim3(nt), smem, stream, dy, x, emb, mean, rstd, dx, sig, kap,
                      S, D, T, keep_dx ? 1 : 0);
}

// 16 columns per thread.  Stages of up to 12 KB (D <= 3072): two CTAs of <= 192
// threads per SM, blocks of 4 rows, 8 stages; up to 16 KB: one CTA of <= 256
// threads per SM, the same ring; longer rows: 32 columns per thread, blocks of
// 2 rows and 4 stages (at most 128 KB).
cudaError_t launch_out_bwd(const uint16_t *dy, const uint16_t *x, const uint16_t *emb, const float *mean,
                           const float *rstd, uint16_t *dx, float *d_emb, void *ws, int B, int S, int D,
                           cudaStream_t stream, const DeviceInfo &dev, bool keep_dx) {
    if (S == 0) return launch_zero(d_emb, (size_t)B * 2 * D, stream);
    const int T = (S + kTile - 1) / kTile;
    const int H = 2 * D;
    float *sig = static_cast<float *>(ws);
    float *kap = sig + (size_t)B * T * H;
    const int V = D / 8;
    cudaError_t err;
    if (V <= 384)
        err = launch_out_bwd_t<2, 192, 2, 4, 8>(dy, x, emb, mean, rstd, dx, sig, kap, B, S, D, T, stream, dev, keep_dx);
    else if (V <= 512)
        err = launch_out_bwd_t<2, 256, 1, 4, 8>(dy, x, emb, mean, rstd, dx, sig, kap, B, S, D, T, stream, dev, keep_dx);
    else
        err = launch_out_bwd_t<4, 256, 1, 2, 4>(dy, x, emb, mean, rstd, dx, sig, kap, B, S, D, T, stream, dev, keep_dx);
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

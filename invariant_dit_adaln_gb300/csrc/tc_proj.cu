// The modulation projection on the tensor cores (tcgen05, TMEM, TMA):
//     emb[b, n] = bf16( sum_k W[n, k] u[b, k]  +  bias[n] ),   u = bf16(silu(temb))
// RL-Kernel PR 538 "final_adaln_out", section "What" (a fixed-order projection),
// and "Scope / Known limitations" (a conditioning batch runs the same code for
// every size).
//
// The weight is the MMA's A operand and the samples its N: a tile is 128 rows
// of W (MMA M) by 32 samples (MMA N; samples past B read as zeros), for every
// B.  k is cut into `ksplit` contiguous ranges, a function of D only (enough
// CTAs to stream W from every SM: 3 for D = 3072); the CTAs of one tile's
// ranges form a thread block cluster.  Within a range, k ascends in blocks of
// 64 (one 128-byte swizzle row of bf16), each block four tcgen05.mma of
// 128 x 32 x 16 accumulating in fp32 in tensor memory.  Each non-leading CTA of
// the cluster writes its partial sums into the leading CTA's shared memory,
// which adds them in range order, ((p0 + p1) + p2) ..., then the bias, and
// rounds once to bf16.  A sample's column depends only on its own row of u and
// on W, never on the other samples of the tile, so emb for a sample has the
// same bits at every B and every position in the batch.  A CTA may run up to
// 8 sample tiles (8 accumulators) against each W stage it loads.
//
// Roles (128 threads): warp 0 lane 0 issues the TMA loads (the W tiles of the
// first stages before the dependency wait: W is an input of this call and the
// kernel before this one, the SiLU kernel, waited for all earlier work before
// letting this one start; u after the wait); warp 1 lane 0 issues the MMAs;
// then thread t reads the accumulator row of feature n0 + t (tcgen05.ld).
// Every wait on a copy or an MMA has a time limit; one that runs out sets this
// file's error word, the kernel lets its issued copies and MMAs finish, frees
// its tensor memory and returns without writing emb.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace adaln {

constexpr int kTcM = 128;                      // rows of W per tile (MMA M)
constexpr int kTcN = 32;                       // samples per tile (MMA N)
constexpr int kTcK = 64;                       // k per block (128 bytes of bf16)
constexpr int kTcMaxStages = 6;
constexpr int kTcMaxNT = 8;                    // sample tiles per CTA (one accumulator each)
constexpr int kTcWTile = kTcM * kTcK * 2;      // 16 KB
constexpr int kTcUTile = kTcN * kTcK * 2;      // 4 KB
constexpr int kTcUTileSmall = 8 * kTcK * 2;    // 1 KB: the u tile of at most 8 samples
constexpr int kTcPartBytes = kTcN * kTcM * 4;  // one accumulator, fp32
constexpr int kTcMaxSplit = 8;                 // portable cluster size
constexpr int kTcSplitTarget = 152;            // CTAs aimed at (ranges fixed by D alone)
constexpr int kTcMaxArea = 200 * 1024;         // stage buffers, one CTA per SM
constexpr int kTcSmallArea = 108 * 1024;       // stage buffers, two CTAs fit on an SM
constexpr int kTcSmemExtra = 256 + 1024;       // barriers, alignment

// bytes of a pipeline stage: kblk k blocks, each a W tile and nt u tiles
__host__ __device__ constexpr int tc_stage_bytes(int kblk, int nt, int utile) {
    return kblk * (kTcWTile + nt * utile);
}

static_assert(kTcWTile % 1024 == 0 && kTcUTile % 1024 == 0, "tiles on 1024-byte swizzle-atom boundaries");
static_assert(kTcN % 16 == 0 && kTcN >= 16 && kTcN <= 256, "MMA N for M = 128");
static_assert(kTcMaxNT * kTcN <= 512, "tensor memory columns");
static_assert(tc_stage_bytes(2, kTcMaxNT, kTcUTile) * 2 <= kTcMaxArea, "two stages at the most sample tiles");
static_assert(tc_stage_bytes(3, 1, kTcUTileSmall) * 2 <= kTcSmallArea, "two stages of three k blocks, <= 8 samples");
static_assert(tc_stage_bytes(2, 2, kTcUTile) * 2 <= kTcSmallArea, "two stages of two k blocks, two sample tiles");
static_assert((kTcMaxSplit - 1) * kTcPartBytes <= kTcMaxArea * 3 / 4,
              "one sample tile's partials fit in the larger stage buffers (at least 3/4 of them hold stages)");
static_assert(kTcMaxArea + kTcSmemExtra <= 227 * 1024, "shared memory");
static_assert(2 * (kTcSmallArea + kTcSmemExtra + 1024) <= 228 * 1024, "two CTAs per SM");

static __device__ unsigned g_err_tc;
__device__ __forceinline__ void report_error_tc(unsigned code) {
    if (code == kErrDrainFailed)
        atomicOr(&g_err_tc, code);
    else
        atomicCAS(&g_err_tc, 0u, code);
}

struct TcSmem {
    uint64_t full[kTcMaxStages];   // a stage's tiles have landed
    uint64_t empty[kTcMaxStages];  // the MMAs reading a stage are done
    uint64_t done;                 // every issued MMA is done
    uint32_t tmem;                 // accumulator address (lane 0, first column)
    int abort;
    int bad[kTcMaxSplit];          // leading CTA: a CTA of the cluster gave up
#ifdef ADALN_TEST_WAIT_NEVER_NS
    uint64_t never;                // test builds: a barrier nothing arrives on
#endif
};
static_assert(sizeof(TcSmem) <= 256, "barrier block");

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzled
// layout: rows of 128 bytes, groups of 8 rows `sbo` bytes apart (the stride
// byte offset: 1024 for a dense tile; 0 makes every group read the first 8
// rows); the leading byte offset is not used by this layout.  Fields: start
// address / 16 (bits 0-13), leading offset / 16 (16-29), stride offset / 16
// (32-45), descriptor version 1 (46-47), swizzle mode 2 = 128 bytes (61-63).
__device__ __forceinline__ uint64_t tc_desc(uint32_t saddr, uint32_t sbo = 1024) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(sbo >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N / 8 in
// bits 17-22, M / 16 in bits 24-28.
constexpr uint32_t kTcIdesc =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kTcN >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_hint(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar,
                                                 uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// address of the same shared-memory location in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ void st_cluster_s32(uint32_t addr, int v) {
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// the kTcN accumulator columns [col, col + kTcN) of this warp's 32 lanes
static_assert(kTcN == 16 || kTcN == 32, "accumulator tile width");
__device__ __forceinline__ void tmem_ld_tile(uint32_t taddr, uint32_t (&v)[kTcN]) {
    if constexpr (kTcN == 32) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
            "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
              "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]),
              "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]),
              "=r"(v[30]), "=r"(v[31])
            : "r"(taddr));
    } else {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
            "%15}, [%16];"
            : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
              "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
            : "r"(taddr));
    }
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// k blocks [kb_begin(r), kb_begin(r + 1)) belong to range r of ksplit
__device__ __forceinline__ int kb_begin(int KB, int ksplit, int r) { return (int)((long long)KB * r / ksplit); }

struct TcArgs {
    const uint16_t *bias;
    uint16_t *emb;
    int B, D;
    int ksplit;     // k ranges (cluster size)
    int nt;         // sample tiles per CTA
    int nstages;    // pipeline stages
    int kblk;       // k blocks per stage
    int area;       // bytes of stage buffers (the barriers follow them)
    int u_rows;     // rows of the u box: B rounded up to 8 below 32 samples, else 32
    int utile;      // bytes of a u tile: 4 KB, or 1 KB (8 rows, read by every row group) for B <= 8
    int red_tiles;  // sample tiles whose partials one round of the cluster reduction moves
    int tmem_cols;  // allocated accumulator columns (power of two >= 32 nt)
};

// Grid: (ksplit, 2D / 128, ceil(B / (32 nt))); the cluster is the ksplit
// CTAs of one (W tile, sample group).
__global__ void __launch_bounds__(128, 1)
proj_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_u,
                   const TcArgs a) {
    extern __shared__ unsigned char tc_smem_raw[];
    const uint32_t raw = smem_u32(tc_smem_raw);
    unsigned char *stages = tc_smem_raw + (((raw + 1023u) & ~1023u) - raw);
    TcSmem &sm = *reinterpret_cast<TcSmem *>(stages + a.area);
    volatile int *abort_flag = &sm.abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int N = 2 * a.D;
    const int nt = a.nt, S = a.nstages;
    const int KS = a.kblk;
    const int stage_bytes = tc_stage_bytes(KS, nt, a.utile);
    const uint32_t u_sbo = a.utile == kTcUTile ? 1024u : 0u;
    const uint32_t rank = cluster_rank();  // == blockIdx.x: the cluster spans the k ranges of one tile
    const int n0 = blockIdx.y * kTcM;
    const int m0 = blockIdx.z * kTcN * nt;
    const int KB = a.D / kTcK;
    const int kb0 = kb_begin(KB, a.ksplit, (int)rank);
    const int nkb = kb_begin(KB, a.ksplit, (int)rank + 1) - kb0;
    const int nst = (nkb + KS - 1) / KS;
    const uint32_t kb_tx = (uint32_t)(kTcWTile + nt * a.u_rows * kTcK * 2);  // bytes of one k block

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.done, 1);
        sm.abort = 0;
        for (int r = 0; r < kTcMaxSplit; ++r) sm.bad[r] = 0;
#ifdef ADALN_TEST_WAIT_NEVER_NS
        mbar_init(&sm.never, 1);
#endif
        fence_barrier_init();
    }
    if (a.utile == kTcUTile && a.u_rows < kTcN) {
        // rows u_rows..31 of every u tile: zeros, read by the MMA, never loaded
        const int per_tile = (kTcN - a.u_rows) * kTcK * 2 / 16;
        const int tiles = S * KS * nt;
        for (int i = threadIdx.x; i < tiles * per_tile; i += blockDim.x) {
            const int t = i / per_tile, j = i - t * per_tile;
            unsigned char *tile = stages + (t / (KS * nt)) * stage_bytes + KS * kTcWTile + (t % (KS * nt)) * a.utile;
            stg16(tile + a.u_rows * kTcK * 2 + j * 16, make_uint4(0u, 0u, 0u, 0u));
        }
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.tmem)),
                     "r"(a.tmem_cols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = sm.tmem;

    // stage i, k block j: the W tile, then the u tiles of the nt sample tiles
    auto w_tile = [&](int s, int j) { return stages + s * stage_bytes + j * kTcWTile; };
    auto u_tile = [&](int s, int j, int t) {
        return stages + s * stage_bytes + KS * kTcWTile + (j * nt + t) * a.utile;
    };

    if (warp == 0 && lane == 0) {
        // ---- producer ----
        const uint64_t pol_w = l2_evict_last();  // the backward projection reads W again
        const int first = min(S, nst);
        for (int i = 0; i < first; ++i) {
            const int nk = min(KS, nkb - i * KS);
            mbar_arrive_expect_tx(&sm.full[i], (uint32_t)nk * kb_tx);
            for (int j = 0; j < nk; ++j)
                tma_load_2d_hint(w_tile(i, j), &map_w, (kb0 + i * KS + j) * kTcK, n0, &sm.full[i], pol_w);
        }
        pdl_wait();  // u comes from the SiLU kernel
        for (int i = 0; i < first; ++i) {
            const int nk = min(KS, nkb - i * KS);
            for (int j = 0; j < nk; ++j)
                for (int t = 0; t < nt; ++t)
                    tma_load_2d(u_tile(i, j, t), &map_u, (kb0 + i * KS + j) * kTcK, m0 + t * kTcN, &sm.full[i]);
        }
        int issued = first;
        for (int i = first; i < nst; ++i) {
            const int s = i % S;
            if (!mbar_wait_or_abort(&sm.empty[s], (uint32_t)(i / S - 1) & 1u, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            const int nk = min(KS, nkb - i * KS);
            mbar_arrive_expect_tx(&sm.full[s], (uint32_t)nk * kb_tx);
            for (int j = 0; j < nk; ++j) {
                const int kc = (kb0 + i * KS + j) * kTcK;
                tma_load_2d_hint(w_tile(s, j), &map_w, kc, n0, &sm.full[s], pol_w);
                for (int t = 0; t < nt; ++t) tma_load_2d(u_tile(s, j, t), &map_u, kc, m0 + t * kTcN, &sm.full[s]);
            }
            issued = i + 1;
        }
        // every copy issued has landed before the CTA may leave (at once when
        // the MMAs consumed them: no later phase of the stage was started)
        for (int s = 0; s < S && s < issued; ++s) {
            const int last = s + S * ((issued - 1 - s) / S);
            if (!mbar_wait_bounded(&sm.full[s], (uint32_t)(last / S) & 1u, 100000000ull))
                report_error_tc(kErrDrainFailed);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer: accumulator t (columns 32t..32t+31) over ascending k ----
        for (int i = 0; i < nst; ++i) {
            const int s = i % S;
#ifdef ADALN_TEST_WAIT_NEVER_NS
            // test builds: the first wait runs out of time
            if (i == 0 && !mbar_wait_bounded(&sm.never, 0u, (uint64_t)(ADALN_TEST_WAIT_NEVER_NS))) {
                *abort_flag = 1;
                break;
            }
#endif
            if (!mbar_wait_or_abort(&sm.full[s], (uint32_t)(i / S) & 1u, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int nk = min(KS, nkb - i * KS);
            // descriptors advance in their address field (bytes / 16): 2 per
            // k slice of 16, utile / 16 per sample tile
            const uint64_t u_step = (uint64_t)(a.utile >> 4);
            for (int j = 0; j < nk; ++j) {
                const uint64_t ad0 = tc_desc(smem_u32(w_tile(s, j)));
                const uint64_t bd0 = tc_desc(smem_u32(u_tile(s, j, 0)), u_sbo);
#pragma unroll
                for (int k = 0; k < kTcK / 16; ++k) {
                    const uint64_t ad = ad0 + 2u * k;
                    const uint32_t accumulate = (i > 0 || j > 0 || k > 0) ? 1u : 0u;
                    uint64_t bd = bd0 + 2u * k;
                    uint32_t acc_addr = tmem;
                    for (int t = 0; t < nt; ++t, bd += u_step, acc_addr += kTcN) {
                        asm volatile(
                            "{\n\t.reg .pred p;\n\t"
                            "setp.ne.b32 p, %4, 0;\n\t"
                            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(acc_addr),
                            "l"(ad), "l"(bd), "r"(kTcIdesc), "r"(accumulate)
                            : "memory");
                    }
                }
            }
            // the stage is free once these MMAs have read it
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_u32(&sm.empty[s]))
                         : "memory");
        }
        // also after giving up: `done` completes when every issued MMA has
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(&sm.done))
                     : "memory");
    }
    pdl_trigger();

    // ---- thread t holds feature n0 + t of every sample in its accumulators ----
    bool ok = mbar_wait_or_abort(&sm.done, 0u, abort_flag) && !*abort_flag;
    if (!ok && threadIdx.x == 0) {
        report_error_tc(kErrProjTcWait);
        // MMAs may still be writing the accumulators
        if (!mbar_wait_bounded(&sm.done, 0u, 100000000ull)) report_error_tc(kErrDrainFailed);
    }
    ok = __syncthreads_and(ok);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);

    // The ranges' partial sums meet in the leading CTA (rank 0), red_tiles
    // sample tiles per round.  After the first cluster barrier the stage
    // buffers of every CTA are free (copies landed, MMAs done); the leader's
    // hold the others' partials of the round.
    float4 *part = reinterpret_cast<float4 *>(stages);  // [ksplit - 1][red_tiles][kTcN / 4][kTcM]
    const int n = n0 + threadIdx.x;
    const float bn = bf16f(a.bias[n]);
    for (int t0 = 0; t0 < nt; t0 += a.red_tiles) {
        const int t1 = min(nt, t0 + a.red_tiles);
        if (a.ksplit > 1) {
            cluster_sync();
            if (rank > 0) {
                for (int t = t0; t < t1; ++t) {
                    uint32_t v[kTcN];
                    tmem_ld_tile(trow + (uint32_t)(t * kTcN), v);
                    float4 *mine = part + ((size_t)(rank - 1) * a.red_tiles + (t - t0)) * (kTcN / 4) * kTcM;
#pragma unroll
                    for (int c = 0; c < kTcN / 4; ++c)
                        st_cluster_v4(map_to_rank(mine + c * kTcM + threadIdx.x, 0),
                                      make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                                  __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3])));
                }
                if (threadIdx.x == 0) st_cluster_s32(map_to_rank(&sm.bad[rank], 0), ok ? 0 : 1);
            }
            cluster_sync();
        }
        if (rank != 0) continue;
        bool all_ok = ok;
        for (int r = 1; r < a.ksplit; ++r) all_ok = all_ok && sm.bad[r] == 0;
        if (!all_ok) continue;
        for (int t = t0; t < t1; ++t) {
            uint32_t v[kTcN];
            tmem_ld_tile(trow + (uint32_t)(t * kTcN), v);
            float acc[kTcN];
#pragma unroll
            for (int c = 0; c < kTcN; ++c) acc[c] = __uint_as_float(v[c]);
            for (int r = 1; r < a.ksplit; ++r) {
                const float4 *theirs = part + ((size_t)(r - 1) * a.red_tiles + (t - t0)) * (kTcN / 4) * kTcM;
#pragma unroll
                for (int c = 0; c < kTcN / 4; ++c) {
                    const float4 p = theirs[c * kTcM + threadIdx.x];
                    acc[4 * c] = __fadd_rn(acc[4 * c], p.x);
                    acc[4 * c + 1] = __fadd_rn(acc[4 * c + 1], p.y);
                    acc[4 * c + 2] = __fadd_rn(acc[4 * c + 2], p.z);
                    acc[4 * c + 3] = __fadd_rn(acc[4 * c + 3], p.w);
                }
            }
            const int mt = m0 + t * kTcN;
#pragma unroll
            for (int c = 0; c < kTcN; ++c)
                if (mt + c < a.B) a.emb[(size_t)(mt + c) * N + n] = bf16_bits(__fadd_rn(acc[c], bn));
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(a.tmem_cols)
                     : "memory");
    }
}

// --------------------------------------------------------------------------
// proj_out (the latent projection 3072 -> 64 after the final norm; RL-Kernel
// PR 538 "What" leaves it to latent_proj_gemm) on the tensor cores, fused with
// the LayerNorm forward in one call: the forward writes out as evict-last in
// L2 and this kernel reads it back from there.
//     y[r, j] = bf16( sum_d out[r, d] Wp[j, d]  +  bp[j] )
// A tile is 128 token rows of out (MMA M) by the 64 rows of Wp (MMA N); k is
// cut into kPoSplit(D) ranges (a cluster, partials added in range order in
// the leading CTA), ascending blocks of 64 within a range, four tcgen05.mma of
// 128 x 64 x 16 per block.  A token's row of y depends only on its own row of
// out, so y does not depend on B, S or the token's position.
// --------------------------------------------------------------------------
constexpr int kPoN = 64;                              // rows of Wp (MMA N)
constexpr int kPoKblk = 2;                            // k blocks per stage
constexpr int kPoStages = 4;
constexpr int kPoATile = kTcM * kTcK * 2;             // 16 KB of out
constexpr int kPoBTile = kPoN * kTcK * 2;             // 8 KB of Wp
constexpr int kPoStageBytes = kPoKblk * (kPoATile + kPoBTile);
constexpr int kPoArea = kPoStages * kPoStageBytes;    // 192 KB
constexpr size_t kPoSmemBytes = (size_t)kPoArea + 256 + 1024;
constexpr uint32_t kPoIdesc =
    (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kPoN >> 3) << 17) | ((uint32_t)(kTcM >> 4) << 24);
static_assert(kPoSmemBytes <= 227 * 1024, "shared memory");
static_assert(kPoN * kTcM * 4 <= kPoArea, "one partner's partials fit in the stage buffers");

struct PoSmem {
    uint64_t full[kPoStages];
    uint64_t empty[kPoStages];
    uint64_t done;
    uint32_t tmem;
    int abort;
    int bad;
#ifdef ADALN_TEST_WAIT_NEVER_NS
    uint64_t never;  // test builds: a barrier nothing arrives on
#endif
};

__global__ void __launch_bounds__(128, 1)
proj_out_tc_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                   const uint16_t *__restrict__ bp, uint16_t *__restrict__ y, int R, int D, int ksplit) {
    extern __shared__ unsigned char po_smem_raw[];
    const uint32_t raw = smem_u32(po_smem_raw);
    unsigned char *stages = po_smem_raw + (((raw + 1023u) & ~1023u) - raw);
    PoSmem &sm = *reinterpret_cast<PoSmem *>(stages + kPoArea);
    volatile int *abort_flag = &sm.abort;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const int r0 = blockIdx.y * kTcM;
    const int KB = D / kTcK;
    const int kb0 = kb_begin(KB, ksplit, (int)rank);
    const int nkb = kb_begin(KB, ksplit, (int)rank + 1) - kb0;
    const int nst = (nkb + kPoKblk - 1) / kPoKblk;
    constexpr uint32_t kb_tx = kPoATile + kPoBTile;

    if (threadIdx.x == 0) {
        for (int st = 0; st < kPoStages; ++st) {
            mbar_init(&sm.full[st], 1);
            mbar_init(&sm.empty[st], 1);
        }
        mbar_init(&sm.done, 1);
        sm.abort = 0;
        sm.bad = 0;
#ifdef ADALN_TEST_WAIT_NEVER_NS
        mbar_init(&sm.never, 1);
#endif
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&sm.tmem)),
                     "r"(kPoN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = sm.tmem;
    auto a_tile = [&](int st, int j) { return stages + st * kPoStageBytes + j * kPoATile; };
    auto b_tile = [&](int st, int j) { return stages + st * kPoStageBytes + kPoKblk * kPoATile + j * kPoBTile; };

    if (warp == 0 && lane == 0) {
        // ---- producer: Wp of the first stages before the wait (a call input;
        // the LayerNorm kernel before this one waited for all earlier work),
        // out after it ----
        const uint64_t pol_a = l2_evict_first();  // out is read once more, here
        const int first = min(kPoStages, nst);
        for (int i = 0; i < first; ++i) {
            const int nk = min(kPoKblk, nkb - i * kPoKblk);
            mbar_arrive_expect_tx(&sm.full[i], (uint32_t)nk * kb_tx);
            for (int j = 0; j < nk; ++j) tma_load_2d(b_tile(i, j), &map_b, (kb0 + i * kPoKblk + j) * kTcK, 0, &sm.full[i]);
        }
        pdl_wait();
        for (int i = 0; i < first; ++i) {
            const int nk = min(kPoKblk, nkb - i * kPoKblk);
            for (int j = 0; j < nk; ++j)
                tma_load_2d_hint(a_tile(i, j), &map_a, (kb0 + i * kPoKblk + j) * kTcK, r0, &sm.full[i], pol_a);
        }
        int issued = first;
        for (int i = first; i < nst; ++i) {
            const int st = i % kPoStages;
            if (!mbar_wait_or_abort(&sm.empty[st], (uint32_t)(i / kPoStages - 1) & 1u, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            const int nk = min(kPoKblk, nkb - i * kPoKblk);
            mbar_arrive_expect_tx(&sm.full[st], (uint32_t)nk * kb_tx);
            for (int j = 0; j < nk; ++j) {
                const int kc = (kb0 + i * kPoKblk + j) * kTcK;
                tma_load_2d(b_tile(st, j), &map_b, kc, 0, &sm.full[st]);
                tma_load_2d_hint(a_tile(st, j), &map_a, kc, r0, &sm.full[st], pol_a);
            }
            issued = i + 1;
        }
        for (int st = 0; st < kPoStages && st < issued; ++st) {
            const int last = st + kPoStages * ((issued - 1 - st) / kPoStages);
            if (!mbar_wait_bounded(&sm.full[st], (uint32_t)(last / kPoStages) & 1u, 100000000ull))
                report_error_tc(kErrDrainFailed);
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        for (int i = 0; i < nst; ++i) {
            const int st = i % kPoStages;
#ifdef ADALN_TEST_WAIT_NEVER_NS
            // test builds: the first wait runs out of time
            if (i == 0 && !mbar_wait_bounded(&sm.never, 0u, (uint64_t)(ADALN_TEST_WAIT_NEVER_NS))) {
                *abort_flag = 1;
                break;
            }
#endif
            if (!mbar_wait_or_abort(&sm.full[st], (uint32_t)(i / kPoStages) & 1u, abort_flag)) {
                *abort_flag = 1;
                break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const int nk = min(kPoKblk, nkb - i * kPoKblk);
            for (int j = 0; j < nk; ++j) {
                const uint64_t ad0 = tc_desc(smem_u32(a_tile(st, j))), bd0 = tc_desc(smem_u32(b_tile(st, j)));
#pragma unroll
                for (int k = 0; k < kTcK / 16; ++k) {
                    const uint32_t accumulate = (i > 0 || j > 0 || k > 0) ? 1u : 0u;
                    asm volatile(
                        "{\n\t.reg .pred p;\n\t"
                        "setp.ne.b32 p, %4, 0;\n\t"
                        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
                        "l"(ad0 + 2u * k), "l"(bd0 + 2u * k), "r"(kPoIdesc), "r"(accumulate)
                        : "memory");
                }
            }
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                             smem_u32(&sm.empty[st]))
                         : "memory");
        }
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         smem_u32(&sm.done))
                     : "memory");
    }
    pdl_trigger();

    bool ok = mbar_wait_or_abort(&sm.done, 0u, abort_flag) && !*abort_flag;
    if (!ok && threadIdx.x == 0) {
        report_error_tc(kErrProjOutWait);
        if (!mbar_wait_bounded(&sm.done, 0u, 100000000ull)) report_error_tc(kErrDrainFailed);
    }
    ok = __syncthreads_and(ok);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    // thread t holds token row r0 + t: columns 0..31 and 32..63 of the accumulator
    uint32_t v[kPoN];
    {
        const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
        uint32_t (&v0)[kTcN] = *reinterpret_cast<uint32_t(*)[kTcN]>(&v[0]);
        uint32_t (&v1)[kTcN] = *reinterpret_cast<uint32_t(*)[kTcN]>(&v[kTcN]);
        tmem_ld_tile(trow, v0);
        tmem_ld_tile(trow + kTcN, v1);
    }
    float4 *part = reinterpret_cast<float4 *>(stages);  // [ksplit - 1][kPoN / 4][kTcM]
    if (ksplit > 1) {
        cluster_sync();
        if (rank > 0) {
            float4 *mine = part + (size_t)(rank - 1) * (kPoN / 4) * kTcM;
#pragma unroll
            for (int c = 0; c < kPoN / 4; ++c)
                st_cluster_v4(map_to_rank(mine + c * kTcM + threadIdx.x, 0),
                              make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                                          __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3])));
            if (threadIdx.x == 0 && !ok) st_cluster_s32(map_to_rank(&sm.bad, 0), 1);
        }
        cluster_sync();
    }
    const int r = r0 + threadIdx.x;
    if (rank == 0 && ok && sm.bad == 0 && r < R) {
        float acc[kPoN];
#pragma unroll
        for (int c = 0; c < kPoN; ++c) acc[c] = __uint_as_float(v[c]);
        for (int q = 1; q < ksplit; ++q) {
            const float4 *theirs = part + (size_t)(q - 1) * (kPoN / 4) * kTcM;
#pragma unroll
            for (int c = 0; c < kPoN / 4; ++c) {
                const float4 p = theirs[c * kTcM + threadIdx.x];
                acc[4 * c] = __fadd_rn(acc[4 * c], p.x);
                acc[4 * c + 1] = __fadd_rn(acc[4 * c + 1], p.y);
                acc[4 * c + 2] = __fadd_rn(acc[4 * c + 2], p.z);
                acc[4 * c + 3] = __fadd_rn(acc[4 * c + 3], p.w);
            }
        }
        uint4 *dst = reinterpret_cast<uint4 *>(y + (size_t)r * kPoN);
#pragma unroll
        for (int c = 0; c < kPoN / 8; ++c) {
            const uint4 bw = ldg16(bp + 8 * c);
            const uint32_t b4[4] = {bw.x, bw.y, bw.z, bw.w};
            uint32_t o[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                o[q] = pack_bf16x2(__fadd_rn(acc[8 * c + 2 * q], bf16lo(b4[q])),
                                   __fadd_rn(acc[8 * c + 2 * q + 1], bf16hi(b4[q])));
            dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    if (warp == 1) {
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kPoN) : "memory");
    }
}

// --------------------------------------------------------------------------
// host side
// --------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// the driver's tensor-map encoder, looked up once through the runtime
static EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// A [rows, cols] bf16 row-major tensor as a TMA map whose boxes are
// box_rows x 64 columns, 128-byte swizzled; elements outside read as zeros.
static bool make_map(CUtensorMap *m, const void *ptr, int rows, int cols, int box_rows) {
    EncodeTiledFn f = encode_fn();
    if (!f) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTcK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool proj_fwd_tc_supported(int D) { return D > 0 && D % kTcK == 0 && encode_fn() != nullptr; }

// The number of k ranges for D: about kTcSplitTarget CTAs over the 2D / 128
// tiles of W, at most a portable cluster and at most one range per k block.
// (On a 152-SM GB300 the clusters of one sample group then run in one wave.)
int proj_fwd_tc_ksplit(int D) {
    const int tiles = 2 * D / kTcM;
    const int KB = D / kTcK;
    int ks = kTcSplitTarget / tiles;
    if (ks > kTcMaxSplit) ks = kTcMaxSplit;
    if (ks > KB) ks = KB;
    return ks < 1 ? 1 : ks;
}

// emb from u (written by the kernel before this one on the stream).  The
// sample tiles per CTA (nt), the u tile layout, the k blocks per stage and the
// pipeline depth change only how the work is scheduled, never the arithmetic
// of a sample's column.  Up to five sample tiles the stage buffers leave room
// for two CTAs on an SM, so that every cluster is resident at once (the 48
// clusters of 3 CTAs of D = 3072 would take two waves at one CTA per SM);
// more samples take the larger buffers, for more reuse of each W stage.
cudaError_t launch_proj_fwd_tc(const uint16_t *u, const uint16_t *W, const uint16_t *bias, uint16_t *emb, int B,
                               int D, cudaStream_t stream, const DeviceInfo &dev) {
    TcArgs a;
    a.bias = bias;
    a.emb = emb;
    a.B = B;
    a.D = D;
    a.ksplit = proj_fwd_tc_ksplit(D);
    a.u_rows = B >= kTcN ? kTcN : (B + 7) / 8 * 8;
    const int tiles_b = (B + kTcN - 1) / kTcN;
    const size_t parts = (size_t)(a.ksplit - 1) * kTcPartBytes;  // one sample tile's partials
    auto stages_of = [](int area, int kblk, int nt, int utile) {
        const int st = area / tc_stage_bytes(kblk, nt, utile);
        return st < kTcMaxStages ? st : kTcMaxStages;
    };
    int nt, kblk, area, utile;
    if (B <= 8)
        nt = 1, kblk = 2, area = kTcSmallArea, utile = kTcUTileSmall;
    else if (tiles_b <= 2)
        nt = tiles_b, kblk = 2, area = kTcSmallArea, utile = kTcUTile;
    else if (tiles_b <= 5)
        nt = tiles_b, kblk = 1, area = kTcSmallArea, utile = kTcUTile;
    else
        nt = tiles_b < kTcMaxNT ? tiles_b : kTcMaxNT, kblk = 2, area = kTcMaxArea, utile = kTcUTile;
    if (area == kTcSmallArea && parts > (size_t)stages_of(area, kblk, nt, utile) * tc_stage_bytes(kblk, nt, utile))
        kblk = 2, area = kTcMaxArea;  // many k ranges (small D): room for the partials
    a.nt = nt;
    a.kblk = kblk;
    a.area = area;
    a.utile = utile;
    a.nstages = stages_of(area, kblk, nt, utile);
    const size_t room = (size_t)a.nstages * tc_stage_bytes(kblk, nt, utile);
    a.red_tiles = parts == 0 ? nt : (int)(room / parts < (size_t)nt ? room / parts : (size_t)nt);
    if (a.nstages < 2 || a.red_tiles < 1) return cudaErrorInvalidConfiguration;
    int cols = 32;
    while (cols < nt * kTcN) cols *= 2;
    a.tmem_cols = cols;
    CUtensorMap map_w, map_u;
    if (!make_map(&map_w, W, 2 * D, D, kTcM) || !make_map(&map_u, u, B, D, a.u_rows)) return cudaErrorInvalidValue;
    cudaError_t err = ensure_smem_attr((const void *)proj_fwd_tc_kernel, (size_t)kTcMaxArea + kTcSmemExtra, dev);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.ksplit, (unsigned)(2 * D / kTcM), (unsigned)((tiles_b + nt - 1) / nt));
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = (size_t)area + kTcSmemExtra;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributePreferredSharedMemoryCarveout;
    attr[1].val.sharedMemCarveout = (unsigned)cudaSharedmemCarveoutMaxShared;
    attr[2].id = cudaLaunchAttributeClusterDimension;
    attr[2].val.clusterDim.x = (unsigned)a.ksplit;
    attr[2].val.clusterDim.y = 1;
    attr[2].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 3;
    return cudaLaunchKernelEx(&cfg, proj_fwd_tc_kernel, map_w, map_u, a);
}

// k ranges of proj_out: two (a cluster of 2) from 16 k blocks on, else one;
// fixed by D alone
static int proj_out_ksplit(int D) { return D / kTcK >= 16 ? 2 : 1; }

bool proj_out_tc_supported(int D, int J) { return J == kPoN && D > 0 && D % kTcK == 0 && encode_fn() != nullptr; }

cudaError_t launch_out_fwd_proj(const uint16_t *x, const uint16_t *emb, const uint16_t *Wp, const uint16_t *bp,
                                uint16_t *out, float *mean, float *rstd, uint16_t *y, int B, int S, int D,
                                float eps, cudaStream_t stream, const DeviceInfo &dev) {
    const int R = B * S;
    CUtensorMap map_a, map_b;
    if (!make_map(&map_a, out, R, D, kTcM) || !make_map(&map_b, Wp, kPoN, D, kPoN)) return cudaErrorInvalidValue;
    cudaError_t err = launch_out_fwd(x, emb, out, mean, rstd, B, S, D, eps, stream, dev, true);
    if (err != cudaSuccess) return err;
    err = ensure_smem_attr((const void *)proj_out_tc_kernel, kPoSmemBytes, dev);
    if (err != cudaSuccess) return err;
    const int ks = proj_out_ksplit(D);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ks, (unsigned)((R + kTcM - 1) / kTcM), 1);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = kPoSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributePreferredSharedMemoryCarveout;
    attr[1].val.sharedMemCarveout = (unsigned)cudaSharedmemCarveoutMaxShared;
    attr[2].id = cudaLaunchAttributeClusterDimension;
    attr[2].val.clusterDim.x = (unsigned)ks;
    attr[2].val.clusterDim.y = 1;
    attr[2].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 3;
    return cudaLaunchKernelEx(&cfg, proj_out_tc_kernel, map_a, map_b, bp, y, R, D, ks);
}

int read_and_clear_tc_error() {
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_err_tc, sizeof(v)) != cudaSuccess) return -1;
    if (v != 0 && cudaMemcpyToSymbol(g_err_tc, &zero, sizeof(zero)) != cudaSuccess) return -1;
    return (int)v;
}

}  // namespace adaln

// Device helpers shared by the kernels of libadaln.so (sm_103a only).
//
// Numerics: the library is compiled with --fmad=false and without fast math;
// every rounding point of the operator is written with an explicit
// round-to-nearest intrinsic (__fadd_rn, __fmul_rn, ...), so no contraction
// or reassociation can change a result.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace adaln {

// --------------------------------------------------------------------------
// limits shared by the host checks and the kernels
// --------------------------------------------------------------------------
constexpr int kMaxD = 8192;
constexpr int kMaxS = 262144;           // 32^3 * 8 tokens: at most 256 level-1 nodes
constexpr int kTile = 32;               // the token tree's fan-out
constexpr int kMaxLevel1 = kMaxS / (kTile * kTile);  // 256
constexpr int kProjSlabRows = 256;      // rows of W per d_silu partial (fixed by D only)
constexpr int kProjKChunk = 256;        // columns of W per projection-backward CTA

// Error word (device side) set by a wait that ran out of time.
enum DeviceError : unsigned {
    kErrNone = 0,
    kErrOutFwdWait = 0x101,
    kErrOutBwdWait = 0x201,
    kErrProjFwdWait = 0x301,
    kErrProjTcWait = 0x302,
    kErrProjOutWait = 0x303,
    kErrDrainFailed = 0x8000,  // or-ed in: an issued copy did not land while leaving
};

// --------------------------------------------------------------------------
// bf16
// --------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16f(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// two floats -> packed bf16x2 (round to nearest even), lo in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}
__device__ __forceinline__ uint16_t bf16_bits(float f) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// a packed bf16x2 word as (lo, hi) floats: exact
__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }
// eager bf16 multiply and add of two bf16 values: the fp32 result rounded once
__device__ __forceinline__ float eager_mul(float a, float b) { return bf16f(bf16_bits(__fmul_rn(a, b))); }
__device__ __forceinline__ float eager_add(float a, float b) { return bf16f(bf16_bits(__fadd_rn(a, b))); }

// --------------------------------------------------------------------------
// packed fp32x2 arithmetic (one instruction for two lanes of work on sm_103a),
// each result rounded to nearest even, like the scalar __f*_rn forms.
//
// Caution: the compiler may merge a packed multiply into a packed add that
// consumes it, giving one rounding where the source asks for two.  Where a
// product must be rounded before it is added (the operator's x_hat * (1 +
// scale) and the token products g * x_hat), the product is taken with the
// scalar __fmul_rn, which --fmad=false keeps separate.
// --------------------------------------------------------------------------
__device__ __forceinline__ float2 f2splat(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 f2add(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 f2mul(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 f2fma(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
// a - b: b * (-1) is exact, so the fused form rounds once, like a subtraction
__device__ __forceinline__ float2 f2sub(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.0f, -1.0f), a); }

// --------------------------------------------------------------------------
// Packed fp32x2 in inline PTX, on a 64-bit register pair {lo, hi}.
//
// Every operation names its rounding (.rn), and PTX never contracts a
// multiply or an add that carries an explicit rounding into a fused
// multiply-add, so a product written here is always rounded before the add
// that consumes it.  On this GPU a packed instruction occupies the FMA pipe for
// two cycles (it does two lanes of work), so packing halves the issue slots of
// fp32 arithmetic without changing its pipe time.
// --------------------------------------------------------------------------
typedef unsigned long long px2;

__device__ __forceinline__ px2 px_add(px2 a, px2 b) {
    px2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ px2 px_sub(px2 a, px2 b) {
    px2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ px2 px_mul(px2 a, px2 b) {
    px2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ px2 px_fma(px2 a, px2 b, px2 c) {
    px2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ px2 px_make(float lo, float hi) {
    px2 d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
    return d;
}
__device__ __forceinline__ px2 px_splat(float a) { return px_make(a, a); }
__device__ __forceinline__ float px_lo(px2 a) {
    float l;
    asm("{.reg .b32 h;\n\tmov.b64 {%0, h}, %1;}" : "=f"(l) : "l"(a));
    return l;
}
__device__ __forceinline__ float px_hi(px2 a) {
    float h;
    asm("{.reg .b32 l;\n\tmov.b64 {l, %0}, %1;}" : "=f"(h) : "l"(a));
    return h;
}
// a packed bf16x2 word (lo in the low half) as the exact fp32 pair, on the
// integer pipe: the low half moved up by a byte permute, the high half masked
__device__ __forceinline__ px2 px_bf16(uint32_t w) {
    px2 d;
    asm("{.reg .b32 l, h;\n\t"
        "prmt.b32 l, %1, 0, 0x1044;\n\t"
        "and.b32 h, %1, 0xFFFF0000;\n\t"
        "mov.b64 %0, {l, h};}"
        : "=l"(d)
        : "r"(w));
    return d;
}
// a pair rounded to a packed bf16x2 word (round to nearest even), lo low
__device__ __forceinline__ uint32_t px_to_bf16x2(px2 a) {
    uint32_t o;
    asm("{.reg .b32 l, h;\n\t"
        "mov.b64 {l, h}, %1;\n\t"
        "cvt.rn.bf16x2.f32 %0, h, l;}"
        : "=r"(o)
        : "l"(a));
    return o;
}
// Knuth's TwoSum on both lanes: t = s + v and the exact error e of that add
// (s + v = t + e); then c += e and s = t.  Seven packed operations.
__device__ __forceinline__ void px_twosum(px2 &s, px2 &c, px2 v) {
    const px2 t = px_add(s, v);
    const px2 bp = px_sub(t, s);
    const px2 e = px_add(px_sub(s, px_sub(t, bp)), px_sub(v, bp));
    c = px_add(c, e);
    s = t;
}

// --------------------------------------------------------------------------
// SiLU rounded to bf16: the nearest bf16 to the fp64 value of t/(1+exp(-t)).
// Computed in fp32 (error below 4 fp32 ulps); when the fp32 value lies within
// 16 fp32 ulps of a bf16 rounding midpoint, or exp(-t) would overflow fp32,
// it is recomputed in fp64 and rounded once from fp64.
// --------------------------------------------------------------------------
__device__ __forceinline__ uint16_t silu_bf16(uint16_t tb) {
    const float t = bf16f(tb);
    const float den = __fadd_rn(1.0f, expf(-t));
    const float s = __fdiv_rn(t, den);
    const int low = (int)(__float_as_uint(s) & 0xFFFFu) - 0x8000;
    if (t < -80.0f || (low <= 16 && low >= -16)) {
        const double td = (double)t;
        const double sd = td / (1.0 + exp(-td));
        return __bfloat16_as_ushort(__double2bfloat16(sd));
    }
    return bf16_bits(s);
}

// SiLU derivative sigma(t) * (1 + t * (1 - sigma(t))) in fp32
__device__ __forceinline__ float dsilu_f32(float t) {
    const float sg = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-t)));
    return __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(t, __fsub_rn(1.0f, sg))));
}

// --------------------------------------------------------------------------
// Neumaier step (the operator's token tree): t = s + v; the part of the
// smaller operand lost in t is added to c; |s| == |v| takes the first branch.
// --------------------------------------------------------------------------
__device__ __forceinline__ void neumaier(float &s, float &c, float v) {
    const float t = __fadd_rn(s, v);
    const float lost = (fabsf(s) >= fabsf(v)) ? __fadd_rn(__fsub_rn(s, t), v)
                                              : __fadd_rn(__fsub_rn(v, t), s);
    c = __fadd_rn(c, lost);
    s = t;
}

// The same step without a branch (Knuth's TwoSum): t = s + v and the exact
// error e of that add, so that s + v = t + e; then c += e.  Neumaier's branch
// also computes the exact error of t (the operand of larger magnitude minus t
// is exact, and adding the other operand to it is exact too), so both give
// the same t and the same c, bit for bit, whenever t is finite.
__device__ __forceinline__ void twosum(float &s, float &c, float v) {
    const float t = __fadd_rn(s, v);
    const float bp = __fsub_rn(t, s);
    const float e = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(v, bp));
    c = __fadd_rn(c, e);
    s = t;
}
__device__ __forceinline__ void twosum2(float2 &s, float2 &c, float2 v) {
    const float2 t = f2add(s, v);
    const float2 bp = f2sub(t, s);
    const float2 e = f2add(f2sub(s, f2sub(t, bp)), f2sub(v, bp));
    c = f2add(c, e);
    s = t;
}

// --------------------------------------------------------------------------
// warp reductions with a fixed butterfly; every lane ends with the same bits
// (each pairwise add is commutative, so partners compute identical values).
// --------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    return v;
}


// --------------------------------------------------------------------------
// shared memory, mbarriers, bulk copies (the TMA engine), PDL
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// make barrier initialisation visible to the async (TMA) proxy
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for a phase of an mbarrier, for at most `limit_ns` nanoseconds.
// Returns false when the time ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or about `hint_ns` nanoseconds pass, instead of returning at once.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// A wait that sleeps between tries (waiting warps take no issue slots) and
// also gives up as soon as *abort is non-zero (another warp of the CTA gave up
// first) or after `limit_ns`.  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity, const volatile int *abort,
                                                   uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 100000u)) return true;
        if (*abort || globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// The same without sleeping between tries: for a thread on the critical path
// of a pipeline whose phases complete by asynchronous arrivals (TMA bytes,
// tensor-core commits).
__device__ __forceinline__ bool mbar_spin_or_abort(uint64_t *bar, uint32_t parity, const volatile int *abort,
                                                   uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort || globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// plain arrival on an mbarrier (release semantics at CTA scope)
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// atomic add on shared memory with acquire-release semantics at CTA scope:
// the caller's earlier accesses are ordered before it, and the accesses of
// the threads whose additions it observes are visible after it.  Returns the
// old value.
__device__ __forceinline__ unsigned smem_add_acq_rel(unsigned *p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_u32(p)), "r"(v) : "memory");
    return old;
}

// order this thread's (and, after an acquire, the CTA's) generic-proxy
// accesses of shared memory before later async-proxy (bulk copy) accesses
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 1-D bulk copy global -> shared through the TMA engine, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// --------------------------------------------------------------------------
// L2 eviction priority.  A step streams its token tensors (x, dy, out, dx:
// hundreds of MB, each read or written once per call) past the weights W
// (37.7 MB at D = 3072), which both projections read.  Streams are marked
// evict-first and W evict-last, so that W read by the forward projection can
// still be in L2 when the backward projection reads it.
// --------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t l2_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// 16-byte read-only global load with an L2 policy
__device__ __forceinline__ uint4 ldg16_hint(const void *p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}
// 16-byte global store with an L2 policy
__device__ __forceinline__ void stg16_hint(void *p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}
// 16-byte fp32 store with an L2 policy
__device__ __forceinline__ void stg16f_hint(void *p, float4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w), "l"(pol)
                 : "memory");
}
// fp32 load with an L2 policy (coherent at L2: reads what an earlier kernel wrote)
__device__ __forceinline__ float ldcg_hint(const float *p, uint64_t pol) {
    float v;
    asm volatile("ld.global.cg.L2::cache_hint.f32 %0, [%1], %2;" : "=f"(v) : "l"(p), "l"(pol));
    return v;
}

// bulk copy global -> shared with an L2 policy (as bulk_g2s)
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
// L2 prefetch with a policy (as bulk_prefetch_l2)
__device__ __forceinline__ void bulk_prefetch_l2_hint(const void *src, uint32_t bytes, uint64_t pol) {
    asm volatile("cp.async.bulk.prefetch.L2.global.L2::cache_hint [%0], %1, %2;" ::"l"(src), "r"(bytes), "l"(pol)
                 : "memory");
}

// Ask the memory system to bring [src, src + bytes) into L2 (no completion
// to wait for).  L2 is the point of coherence, so this is safe even while the
// preceding kernel may still write the range: later reads see its writes.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// named barrier over `count` threads (a multiple of 32)
__device__ __forceinline__ void named_bar(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Programmatic dependent launch: wait for the preceding grid's completion
// (and the visibility of its writes); allow the next grid to start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// 16-byte global loads/stores
__device__ __forceinline__ uint4 ldg16(const void *p) { return __ldg(reinterpret_cast<const uint4 *>(p)); }
__device__ __forceinline__ void stg16(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }
__device__ __forceinline__ void stg16f(void *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }

}  // namespace adaln

/*
 * adaln.h — C ABI of libadaln.so: the batch-invariant DiT AdaLN final
 * modulation ("norm_out"), forward and backward, on NVIDIA GB300 (sm_103a).
 *
 * The operator (RL-Kernel PR 538 "final_adaln_out", section "What"):
 *
 *     scale, shift = (SiLU(temb) @ W^T + b).chunk(2)      3072 -> 6144, scale first
 *     out          = LayerNorm(x, eps, no affine) * (1 + scale) + shift
 *
 * with the autocast rounding points of miles_diffusion PR 108 ("bitwise
 * train<->rollout parity ...", Summary, root cause 1): LayerNorm computed and
 * returned in fp32, (1 + scale) rounded once to bf16, the modulation in fp32,
 * one bf16 rounding at the store.  The backward returns dx, the token sums
 * d_scale/d_shift through a fixed 32-way Neumaier tree whose shape depends only
 * on the sequence length (PR 538, "What" and the review thread on the
 * cancellation case), and dW, db, d_temb.
 *
 * Every result is bitwise independent of the batch size, of the position of a
 * sample in the batch and (for dW/db) of how samples are split into calls.
 *
 * Conventions for every entry point:
 *  - Pointers are device pointers (memory the current device can read or
 *    write), each 16-byte aligned.  A pointer may be NULL exactly when its
 *    buffer has zero bytes (B == 0 or S == 0), and for the optional outputs
 *    marked "or NULL".  bf16 tensors are passed as their 16-bit
 *    patterns (adaln_bf16); all tensors are dense, row-major, no strides.
 *  - The caller owns every buffer, including workspaces.  A workspace's
 *    contents on entry do not matter (no call needs it zeroed) and are
 *    undefined on return.  The library never
 *    allocates, never frees and never synchronizes: work is enqueued on
 *    `stream` (a cudaStream_t; NULL = the legacy default stream) and the call
 *    returns at once.  Kernels may be launched with programmatic dependent
 *    launch, so a later kernel on the same stream can start its prologue early;
 *    it still reads results only after this call's kernels have completed.
 *  - Outputs must not overlap any input, any other output or the workspace
 *    (ADALN_ERR_ALIAS).  An output is always written, even when it equals an
 *    input value (S == 1 writes a fresh d_emb; nothing is returned as a view).
 *  - All arguments are checked on the host before anything is launched, in
 *    this order: shapes and other argument values, NULL pointers, alignment,
 *    overlaps, workspace, then the current device (must be compute capability
 *    10.3).  A failed check
 *    launches nothing and returns its status.  A failed launch returns
 *    ADALN_ERR_CUDA; an asynchronous device-side fault surfaces, as for any
 *    CUDA work, at the caller's next synchronizing CUDA call.
 *  - Shapes: D % 8 == 0 and 8 <= D <= 8192; 0 <= S <= 262144; B >= 0 with
 *    B <= 65535 for the token-row calls (adaln_out_*, token_sum_tree) and
 *    B <= 2^20 for the projection calls; B * S * D < 2^40.  B == 0 or
 *    S == 0 is valid (see each call).
 *  - Nothing is thrown across the ABI; no global state changes except the
 *    device-side error words read by adaln_device_error() and the per-device
 *    SiLU table filled once by the first adaln_proj_fwd.
 */
#ifndef ADALN_H
#define ADALN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t adaln_bf16; /* bfloat16 bit pattern */

typedef enum adaln_status {
    ADALN_OK = 0,
    ADALN_ERR_NULL = 1,      /* a required pointer is NULL                          */
    ADALN_ERR_SHAPE = 2,     /* a size is out of range (see the conventions)        */
    ADALN_ERR_ALIGN = 3,     /* a pointer is not 16-byte aligned                    */
    ADALN_ERR_ALIAS = 4,     /* an output overlaps an input, output or workspace    */
    ADALN_ERR_WORKSPACE = 5, /* workspace NULL or smaller than the *_workspace_bytes */
    ADALN_ERR_DEVICE = 6,    /* no current CUDA device, or it is not sm_103         */
    ADALN_ERR_CUDA = 7,      /* a CUDA runtime call or a kernel launch failed       */
    ADALN_ERR_ARG = 8        /* another argument is invalid (eps, flag combination) */
} adaln_status;

/* Human-readable name of a status code (static string, never NULL). */
const char *adaln_status_string(int status);

/* ABI version: (major << 16) | minor. */
int adaln_version(void);

/* ------------------------------------------------------------------------ */
/* Forward                                                                    */
/* ------------------------------------------------------------------------ */

/*
 * adaln_proj_fwd — modulation projection (PR 538 "What": the (scale, shift)
 * projection 3072 -> 6144).
 *
 *   u[b,k]   = bf16(silu(temb[b,k]))       the bf16 nearest to the fp64 value of
 *                                          t / (1 + exp(-t))
 *   emb[b,n] = bf16( sum_k u[b,k] * W[n,k]  +  bias[n] )   fp32 accumulation in a
 *              fixed order over k, bias added in fp32, one bf16 rounding
 *
 *   temb [B, D]    bf16   conditioning vector
 *   W    [2D, D]   bf16   row n = output feature n; rows 0..D-1 give scale,
 *                         rows D..2D-1 give shift
 *   bias [2D]      bf16
 *   emb  [B, 2D]   bf16   output, [scale | shift] per sample
 *   u    [B, D]    bf16   output, the SiLU activation (the projection's input,
 *                         saved for adaln_proj_bwd)
 *
 * The k-order of every dot product is fixed by D alone, so emb[b,:] does not
 * depend on B or on b.  For D a multiple of 64 the sum runs on the tensor
 * cores (tcgen05.mma, 128 rows of W x 32 samples x 16 k per instruction,
 * fp32 accumulation in tensor memory): k is cut into a number of contiguous
 * ranges fixed by D (3 for D = 3072), each range summed in ascending blocks
 * of 16, and the ranges' partial sums are added in range order.  Other D use
 * CUDA cores in one fixed order.  B == 0 launches nothing.
 *
 * The first call with B > 0 on a device also fills a 128 KB SiLU lookup table
 * in the library's device memory (a kernel on `stream`) and synchronizes
 * `stream` once; make that first call outside stream capture.  Later calls
 * neither synchronize nor touch the table's contents.
 */
adaln_status adaln_proj_fwd(const adaln_bf16 *temb, const adaln_bf16 *W, const adaln_bf16 *bias,
                            adaln_bf16 *emb, adaln_bf16 *u, int B, int D, void *stream);

/*
 * adaln_out_fwd — LayerNorm (no affine) + modulation (PR 538 "What"; rounding
 * points of PR 108 Summary, root cause 1).
 *
 *   per token row r = (b, s), over d in [0, D):
 *     mean[r] = fp32 sum_d x / D                    fixed-order fp32 reductions
 *     rstd[r] = 1 / sqrt(sum_d (x - mean)^2 / D + eps)   (biased variance)
 *     xhat    = fp32(fp32(x - mean) * rstd)
 *     onep    = bf16(fp32(1 + scale[b,d]))          scale = emb[b, 0:D]
 *     out     = bf16( fp32( fp32(xhat * onep) + shift[b,d] ) )   shift = emb[b, D:2D]
 *
 *   x    [B, S, D] bf16    input tokens
 *   emb  [B, 2D]   bf16    from adaln_proj_fwd
 *   out  [B, S, D] bf16    output
 *   mean [B, S]    fp32    output, saved for the backward
 *   rstd [B, S]    fp32    output, saved for the backward
 *   eps            fp32    LayerNorm epsilon (1e-6 in the model), finite, >= 0
 *
 * The reduction order over d depends only on D; rows never interact.
 * B * S == 0 launches nothing.
 */
adaln_status adaln_out_fwd(const adaln_bf16 *x, const adaln_bf16 *emb, adaln_bf16 *out,
                           float *mean, float *rstd, int B, int S, int D, float eps, void *stream);

/* ------------------------------------------------------------------------ */
/* Backward                                                                   */
/* ------------------------------------------------------------------------ */

/* Workspace bytes adaln_out_bwd needs: the level-0 token-tree partials,
 * 2 * B * ceil(S/32) * 2D fp32 values, rounded up to 256 bytes.  0 if B*S == 0. */
size_t adaln_out_bwd_workspace_bytes(int B, int S, int D);

/*
 * adaln_out_bwd — backward of adaln_out_fwd for the upstream gradient dy
 * (PR 538 "What": LayerNorm backward per row; d_scale, d_shift as token sums
 * in the fixed 32-way tree).
 *
 *   g     = fp32(dy);  gh = g * onep (exact unless it underflows);  xhat as in
 *           the forward, from the saved mean/rstd, bit-identical to the
 *           forward's value
 *   dx    = bf16( rstd * ((gh - c1) - xhat * c2) ),  c1 = sum_d g*onep / D,
 *           c2 = sum_d fp32(g*xhat)*onep / D   (fixed-order fp32 reductions
 *           over d, each sum times the correctly rounded 1/D).  The same
 *           quantity is evaluated as rstd*gh + (mean*k2 - rstd*c1) - x*k2 with
 *           k2 = rstd^2*c2, one multiply and two fused multiply-adds per
 *           element, so dx is within the rounding error of this formula, not
 *           bit-identical to one fixed evaluation of it.
 *   d_emb[b, 0:D]  = d_scale = tree_s( fp32(g * xhat) )
 *   d_emb[b, D:2D] = d_shift = tree_s( g )
 *
 *   tree_s: the fixed 32-way tree over s = 0..S-1.  Level 0 cuts the tokens
 *   into tiles of 32 (the last may be short); each tile is a Neumaier sum in
 *   ascending order starting from its first token, giving (sum, correction).
 *   Each further level cuts the nodes into groups of 32 (the last may be
 *   short); a group's sum is the Neumaier sum of its children's sums in
 *   ascending order, and its correction is that sum's compensation plus the
 *   children's corrections added in ascending order.  The root is the first
 *   level with one node; the result is sum + correction (one IEEE add).  The
 *   shape depends on S only.  Neumaier step: t = s + v; if |s| >= |v| then
 *   c += (s - t) + v else c += (v - t) + s; s = t.
 *
 *   dy, x     [B, S, D] bf16     inputs
 *   emb       [B, 2D]   bf16     input (as given to the forward)
 *   mean,rstd [B, S]    fp32     inputs, from adaln_out_fwd
 *   dx        [B, S, D] bf16     output
 *   d_emb     [B, 2D]   fp32     output, [d_scale | d_shift]
 *   workspace                    >= adaln_out_bwd_workspace_bytes(B, S, D)
 *
 * S == 0 writes d_emb = +0; B == 0 launches nothing.
 */
adaln_status adaln_out_bwd(const adaln_bf16 *dy, const adaln_bf16 *x, const adaln_bf16 *emb,
                           const float *mean, const float *rstd, adaln_bf16 *dx, float *d_emb,
                           void *workspace, size_t workspace_bytes, int B, int S, int D, void *stream);

/*
 * adaln_out_bwd_noalloc — adaln_out_bwd for callers that cannot allocate
 * device memory.  Arguments are checked as for adaln_out_bwd, in the same
 * order (sizes, with the array's limit below counted as a size; NULL pointers;
 * alignment; overlaps; then the device), and only then is the array looked up.  The pages have no counterpart of this call; it exists for
 * code that runs where allocation is not allowed: a plugin inside an engine
 * that owns all device memory and forbids allocations in its execute hook, a
 * real-time loop that must not take the allocator's locks or risk its
 * implicit synchronisation, or a caller with a memory budget fixed at
 * start-up.
 *
 * Same arguments, checks, kernels and results (bit for bit) as
 * adaln_out_bwd, without the workspace: what adaln_out_bwd keeps in its
 * workspace lives in a 24 MiB array inside the library, held on every GPU
 * that loads the library until the process exits.  The call allocates nothing.
 *
 *   Limit: adaln_out_bwd_workspace_bytes(B, S, D) <= 24 MiB = 25165824 bytes
 *   (at D = 3072: B = 2 with S <= 8192, or B = 1 with S <= 16384).  Larger
 *   sizes return ADALN_ERR_SHAPE before anything is launched.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array: two calls whose kernels overlap on
 * the GPU (different streams, no ordering between them) race on it and give
 * wrong results.  Nothing in the array needs to start at zero: every partial
 * the tree reads is written earlier in the same call.
 */
adaln_status adaln_out_bwd_noalloc(const adaln_bf16 *dy, const adaln_bf16 *x, const adaln_bf16 *emb,
                                   const float *mean, const float *rstd, adaln_bf16 *dx, float *d_emb,
                                   int B, int S, int D, void *stream);

/* Workspace bytes token_sum_tree needs: 2 * B * ceil(S/32) * H fp32 values,
 * rounded up to 256 bytes.  0 if B*S == 0. */
size_t token_sum_tree_workspace_bytes(int B, int S, int H);

/*
 * token_sum_tree — the fixed 32-way token tree on its own (PR 538 "What":
 * the FP32 token-sum kernel; review thread on the cancellation case).
 *
 *   out[b,h] = tree_s(in[b,s,h]), the tree defined under adaln_out_bwd.
 *
 *   in  [B, S, H] fp32   H % 4 == 0, 4 <= H <= 2^20
 *   out [B, H]    fp32   output (a fresh buffer, also when S == 1)
 *
 * On the same values it returns the same bytes as the d_emb of
 * adaln_out_bwd.  S == 0 writes out = +0; B == 0 launches nothing.
 */
adaln_status token_sum_tree(const float *in, float *out, int B, int S, int H,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes adaln_proj_bwd needs: the per-slab d_silu partials,
 * ceil(2D/256) * B * D fp32 values, rounded up to 256 bytes. */
size_t adaln_proj_bwd_workspace_bytes(int B, int D);

/*
 * adaln_proj_bwd — backward of adaln_proj_fwd (PR 538 "What": the projection
 * backward of the reused fixed-order projection; the SiLU VJP as in the review
 * finding on the analytic SiLU derivative).
 *
 *   e[b,n]      = bf16(d_emb[b,n])        (emb is a bf16 tensor)
 *   d_temb[b,k] = bf16( (sum_n e[b,n] W[n,k]) * sigma(t) (1 + t (1 - sigma(t))) ),
 *                 t = temb[b,k]; fp32 sum whose n-order is fixed by D alone
 *   dW[n,k]     : acc = accumulate ? dW_acc[n,k] : +0;
 *                 for b = 0 .. B-1 (ascending): acc = acc + e[b,n] * u[b,k]
 *                 (the product is exact in fp32; one rounding per add)
 *   db[n]       : the same with e[b,n] alone
 *
 *   d_emb  [B, 2D] fp32   input (from adaln_out_bwd)
 *   temb   [B, D]  bf16   input
 *   u      [B, D]  bf16   input, the SiLU activation from adaln_proj_fwd
 *   W      [2D, D] bf16   input
 *   d_temb [B, D]  bf16   output
 *   dW_acc [2D, D] fp32   in/out accumulator, or NULL
 *   db_acc [2D]    fp32   in/out accumulator, or NULL
 *   dW     [2D, D] bf16   output bf16(acc), or NULL
 *   db     [2D]    bf16   output bf16(acc), or NULL
 *   accumulate            0: start from +0; 1: start from dW_acc/db_acc (which
 *                         must then be non-NULL for every gradient computed)
 *   workspace             >= adaln_proj_bwd_workspace_bytes(B, D)
 *
 * The weight gradient is computed when dW_acc or dW is non-NULL, the bias
 * gradient when db_acc or db is non-NULL.  Calling with samples 0..k-1 and
 * then, with accumulate = 1, samples k..B-1 gives the same bytes as one call
 * with all B samples.  B == 0 with accumulate = 0 writes zeros.
 */
adaln_status adaln_proj_bwd(const float *d_emb, const adaln_bf16 *temb, const adaln_bf16 *u,
                            const adaln_bf16 *W, adaln_bf16 *d_temb, float *dW_acc, float *db_acc,
                            adaln_bf16 *dW, adaln_bf16 *db, int accumulate,
                            void *workspace, size_t workspace_bytes, int B, int D, void *stream);

/*
 * adaln_proj_wgrad_rows — the weight and bias gradient of adaln_proj_bwd for
 * the output rows n0 <= n < n1 only, over B samples given in ascending order
 * (the projection's dW/db, sharded by output rows: miles_diffusion PR 108,
 * second rendering, "Patches": bitwise parity holds when no partial sums are
 * reduced across GPUs, so a data-parallel step gathers the samples' d_emb and
 * u, and each rank sums all samples for its own rows).
 *
 *   for n0 <= n < n1, with r = n - n0:
 *     dW[r,k] : acc = accumulate ? dW_acc[r,k] : +0;
 *               for b = 0 .. B-1 (ascending): acc = acc + e[b,n] * u[b,k]
 *     db[r]   : the same with e[b,n] alone,      e = bf16(d_emb)
 *
 *   d_emb  [B, 2D]      fp32   input, every sample's (in the global order)
 *   u      [B, D]       bf16   input, the same samples' SiLU activations
 *   dW_acc [n1-n0, D]   fp32   in/out accumulator, or NULL
 *   db_acc [n1-n0]      fp32   in/out accumulator, or NULL
 *   dW     [n1-n0, D]   bf16   output bf16(acc), or NULL
 *   db     [n1-n0]      bf16   output bf16(acc), or NULL
 *
 * The bytes equal rows n0..n1 of adaln_proj_bwd's results on the same samples
 * (the same sequential fp32 order), so concatenating the row blocks of all
 * ranks gives the one-GPU gradient.  0 <= n0 <= n1 <= 2D; no workspace.
 */
adaln_status adaln_proj_wgrad_rows(const float *d_emb, const adaln_bf16 *u, int n0, int n1, float *dW_acc,
                                   float *db_acc, adaln_bf16 *dW, adaln_bf16 *db, int accumulate, int B, int D,
                                   void *stream);

/*
 * adaln_out_fwd_proj — the forward of adaln_out_fwd with the model's next
 * operation, proj_out (the latent projection D -> J = 64 that RL-Kernel PR 538
 * "What" leaves to latent_proj_gemm), in the same call:
 *
 *   out, mean, rstd = adaln_out_fwd(x, emb)        (bits identical to it)
 *   y[b,s,j] = bf16( sum_d out[b,s,d] * Wp[j,d]  +  bp[j] )
 *
 * The sum runs on the tensor cores (tcgen05.mma, 128 token rows x 64 x 16 per
 * instruction, fp32 accumulation in tensor memory): k is cut into a number of
 * contiguous ranges fixed by D (2 from D = 1024 on, else 1), each summed in
 * ascending blocks of 16, the ranges added in order, then the bias, one bf16
 * rounding.  A token's row of y depends only on its row of out.  out stays in
 * L2 (evict-last) between the two kernels.
 *
 *   x [B,S,D], emb [B,2D], Wp [J,D], bp [J] bf16 in;  out [B,S,D], y [B,S,J]
 *   bf16 and mean, rstd [B,S] fp32 out.  D a multiple of 64; J == 64;
 *   B * S <= 65535 * 128.  Errors as adaln_out_fwd; ADALN_ERR_CUDA also when
 *   the driver offers no tensor-map encoder.
 */
adaln_status adaln_out_fwd_proj(const adaln_bf16 *x, const adaln_bf16 *emb, const adaln_bf16 *Wp,
                                const adaln_bf16 *bp, adaln_bf16 *out, float *mean, float *rstd, adaln_bf16 *y,
                                int B, int S, int D, int J, float eps, void *stream);

/* ------------------------------------------------------------------------ */
/* FP32 execution dtype                                                       */
/* ------------------------------------------------------------------------ */

/*
 * The same operator on fp32 tensors (RL-Kernel PR 538 "Results": the FP32
 * timings and the BF16/FP32 acceptance gates): fp32 inputs and outputs, no
 * bf16 rounding anywhere, each step of the eager fp32 graph rounded once to
 * fp32, no TF32.  D is a multiple of 8 up to 4096; otherwise the conventions,
 * checks and errors of the bf16 calls above.
 *
 * adaln_f32_proj_fwd:
 *   u[b,k]   = fp32(silu(t))  (computed in fp64, rounded once)
 *   emb[b,n] = fp32 sum_k u W + bias: lane l of a warp takes the 4-float
 *              vectors l, l+32, ... of row n in ascending order, one fused
 *              multiply-add per element, then a fixed xor butterfly; the
 *              bias added in fp32.  The order depends on D only.
 *   temb [B,D], W [2D,D], bias [2D] fp32 in;  emb [B,2D], u [B,D] fp32 out.
 */
adaln_status adaln_f32_proj_fwd(const float *temb, const float *W, const float *bias, float *emb, float *u, int B,
                                int D, void *stream);

/*
 * adaln_f32_out_fwd:  per row, mean = sum / D, rstd = 1 / sqrt(sum (x -
 * mean)^2 / D + eps) (fixed-order fp32 sums), xhat = fp32(fp32(x - mean) *
 * rstd), onep = fp32(1 + scale), out = fp32(fp32(xhat * onep) + shift).
 *   x [B,S,D], emb [B,2D] fp32 in;  out [B,S,D], mean, rstd [B,S] fp32 out.
 */
adaln_status adaln_f32_out_fwd(const float *x, const float *emb, float *out, float *mean, float *rstd, int B, int S,
                               int D, float eps, void *stream);

/* Workspace bytes adaln_f32_out_bwd needs (the tree nodes, as for adaln_out_bwd). */
size_t adaln_f32_out_bwd_workspace_bytes(int B, int S, int D);

/*
 * adaln_f32_out_bwd:  g = dy, gh = fp32(g * onep); c1 = (sum_d fma g onep) / D,
 * c2 = (sum_d fma p onep) / D with p = fp32(g * xhat); dx = fp32(rstd *
 * ((gh - c1) - xhat * c2)), each operation rounded once; d_emb = [sum_s p |
 * sum_s g] by the fixed 32-way token tree (as adaln_out_bwd, with xhat
 * recomputed from the saved mean and rstd).
 *   dy, x [B,S,D], emb [B,2D], mean, rstd [B,S] fp32 in;  dx [B,S,D], d_emb
 *   [B,2D] fp32 out.
 */
adaln_status adaln_f32_out_bwd(const float *dy, const float *x, const float *emb, const float *mean,
                               const float *rstd, float *dx, float *d_emb, void *workspace, size_t workspace_bytes,
                               int B, int S, int D, void *stream);

/* Workspace bytes adaln_f32_proj_bwd needs: ceil(2D/256) * B * D fp32
 * partials, rounded up to 256 bytes. */
size_t adaln_f32_proj_bwd_workspace_bytes(int B, int D);

/*
 * adaln_f32_proj_bwd:  e = d_emb (no rounding);
 *   d_temb[b,k] = fp32(d_silu * silu'(t)), d_silu = fp32 sum over n of e W in
 *                 slabs of 256 rows (fused multiply-adds, rows ascending),
 *                 the slabs added in ascending order; the product with
 *                 silu'(t) in fp64, rounded once
 *   dW_acc[n,k] : acc = accumulate ? dW_acc : +0; for b ascending:
 *                 acc = fma(e[b,n], u[b,k], acc)   (one rounding per sample)
 *   db_acc[n]   : the same with acc = acc + e[b,n]
 *   d_emb [B,2D], temb, u [B,D], W [2D,D] fp32 in;  d_temb [B,D] out;
 *   dW_acc [2D,D], db_acc [2D] fp32 in/out (either may be NULL).
 */
adaln_status adaln_f32_proj_bwd(const float *d_emb, const float *temb, const float *u, const float *W, float *d_temb,
                                float *dW_acc, float *db_acc, int accumulate, void *workspace,
                                size_t workspace_bytes, int B, int D, void *stream);

/* ------------------------------------------------------------------------ */
/* Block-level modulated norm with a gated residual                           */
/* ------------------------------------------------------------------------ */

/*
 * adaln_scale_residual_norm_fwd — ScaleResidualLayerNormScaleShift, the
 * norm1/norm2 site of every transformer block, with the final norm's rounding
 * points (miles_diffusion PR 108, Summary, root cause 1, and "Patches": fp32
 * LayerNorm, (1 + scale) rounded once to bf16, fp32 modulation; the residual
 * stream's gated add in eager bf16, each operation computed in fp32 and
 * rounded once to bf16).
 *
 *   r[b,s,d]  = bf16( residual[b,s,d] + bf16(gate[b,d] * x[b,s,d]) )
 *   out, mean, rstd = adaln_out_fwd(r, emb)   (the same formulas and orders)
 *
 *   x        [B, S, D] bf16   the branch output (attention or MLP)
 *   residual [B, S, D] bf16   the residual stream
 *   gate     [B, D]    bf16   per-sample gate, broadcast over tokens
 *   emb      [B, 2D]   bf16   [scale | shift] of the block's modulation
 *   r        [B, S, D] bf16   output: the new residual stream (also the
 *                             LayerNorm's input, saved for the backward)
 *   out      [B, S, D] bf16   output
 *   mean, rstd [B, S]  fp32   output, saved for the backward
 *
 * The plain LayerNormScaleShift (no residual) is adaln_out_fwd with the
 * block's [scale | shift] as emb.  Rows never interact.  B * S == 0 launches
 * nothing.  Errors as adaln_out_fwd.
 */
adaln_status adaln_scale_residual_norm_fwd(const adaln_bf16 *x, const adaln_bf16 *residual, const adaln_bf16 *gate,
                                           const adaln_bf16 *emb, adaln_bf16 *r, adaln_bf16 *out, float *mean,
                                           float *rstd, int B, int S, int D, float eps, void *stream);

/* Workspace bytes adaln_scale_residual_norm_bwd needs (the tree nodes of
 * d_scale, d_shift and then of d_gate, in the same space): the same as
 * adaln_out_bwd_workspace_bytes(B, S, D). */
size_t adaln_scale_residual_norm_bwd_workspace_bytes(int B, int S, int D);

/*
 * adaln_scale_residual_norm_bwd — backward of adaln_scale_residual_norm_fwd
 * (autograd of the same graph, with the token sums of the broadcast
 * operands by the fixed 32-way tree of RL-Kernel PR 538 "What").
 *
 *   dr_ln, d_emb = adaln_out_bwd(d_out, r, emb, mean, rstd)
 *   gr[b,s,d]    = bf16(dr_ln + d_r)       (r's two uses; dr_ln if d_r is NULL)
 *   d_residual   = gr
 *   d_x          = bf16(gr * gate)
 *   d_gate[b,d]  = sum over s of bf16(gr * x), fp32, by the token tree
 *
 *   d_out      [B, S, D] bf16   input: the gradient of out
 *   d_r        [B, S, D] bf16   input: the gradient of r from its later uses,
 *                               or NULL (none)
 *   x, r, gate, emb, mean, rstd  inputs as saved by the forward
 *   d_x        [B, S, D] bf16   output
 *   d_residual [B, S, D] bf16   output (it holds dr_ln between the kernels)
 *   d_emb      [B, 2D]   fp32   output [d_scale | d_shift]
 *   d_gate     [B, D]    fp32   output
 *   workspace  >= adaln_scale_residual_norm_bwd_workspace_bytes(B, S, D)
 *
 * Every per-sample output of sample b depends only on sample b.  S == 0
 * writes zero d_emb and d_gate; B == 0 launches nothing.  Outputs may not
 * overlap inputs, each other or the workspace.
 */
adaln_status adaln_scale_residual_norm_bwd(const adaln_bf16 *d_out, const adaln_bf16 *d_r, const adaln_bf16 *x,
                                           const adaln_bf16 *r, const adaln_bf16 *gate, const adaln_bf16 *emb,
                                           const float *mean, const float *rstd, adaln_bf16 *d_x,
                                           adaln_bf16 *d_residual, float *d_emb, float *d_gate, void *workspace,
                                           size_t workspace_bytes, int B, int S, int D, void *stream);

/* ------------------------------------------------------------------------ */
/* Diagnostics                                                                */
/* ------------------------------------------------------------------------ */

/*
 * adaln_device_error — reads and clears the device-side error words of the
 * current device (synchronizes the device).  Kernels that wait on their own
 * asynchronous copies give each wait a time limit; a wait that runs out sets
 * a word instead of hanging, the kernel lets the copies it issued land, and it
 * returns without finishing its outputs.  Codes: 0x101 adaln_out_fwd, 0x201
 * adaln_out_bwd, 0x301 and 0x302 adaln_proj_fwd (CUDA-core and tensor-core
 * kernels), 0x303 adaln_out_fwd_proj (the first code found, LayerNorm kernels
 * first, when several kernels failed); bit 0x8000 is or-ed in when an issued
 * copy did not land within the limit while the kernel was leaving.  Returns 0
 * when no kernel failed, -1 if a word could not be read.
 *
 * Per-device state.  The library keeps, per device ordinal, the SiLU table's
 * readiness, the address of adaln_out_bwd_noalloc's array and the kernels'
 * shared-memory attributes.  cudaDeviceReset (or any other way of replacing a
 * device's primary context) invalidates them: after it, the process must not
 * call the library again on that device.
 */
int adaln_device_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ADALN_H */

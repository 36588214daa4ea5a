/*
 * fp8fg.h -- C ABI of libfp8fg.so: fine-grained FP8 quantisation and the
 * block-scaled FP8 GEMM with per-128-K FP32 promotion, for NVIDIA B300
 * (sm_103a).
 *
 * The operations are those of the FP8 mixed-precision framework of the
 * DeepSeek-V3 Technical Report, section 3.3 (FP8 Training):
 *   - every GEMM operand (Fprop, Dgrad, Wgrad) is E4M3 (section 3.3.1);
 *   - activations are quantised per 1x128 tile and weights per 128x128
 *     block, each group with its own FP32 scale amax/448 (section 3.3.2,
 *     fine-grained quantization);
 *   - the scales run along the GEMM inner dimension K, and each 128-wide K
 *     interval's tensor-core partial sum is promoted to FP32 with the two
 *     scales applied (section 3.3.2, increasing accumulation precision,
 *     Figure 7(b));
 *   - the Wgrad GEMM consumes activations cached in FP8, which needs the
 *     transposed 128x1 grouping along tokens (sections 3.3.1 and 3.3.3; the
 *     report's hardware suggestions in section 3.5.2 note that fusing the
 *     transposition into the GEMM is awkward, so it lives in the quantiser);
 *   - MoE experts run a grouped GEMM over variable per-expert token counts,
 *     which is memory bound at decode batch sizes (section 3.4.2 Decoding).
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers into memory the caller owns.  The library
 *     allocates nothing, frees nothing and keeps no state beyond a per-device
 *     cache of the SM count and per-context caches of kernel attributes and
 *     of the device address of its scratch array (each entry is tagged with
 *     the id of the CUDA context it was made in and is remade when another
 *     context of that device is current).  The caches are guarded by a mutex:
 *     concurrent first calls from several host threads are safe.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls
 *     are asynchronous on that stream and never synchronise, except
 *     fp8_device_error().
 *   - The GEMM entry points launch with programmatic stream serialisation:
 *     their CTAs may start setting up (barriers, tensor memory) while the
 *     kernel before them on the stream finishes, and read nothing from
 *     global memory until that kernel has completed.  Stream order, as the
 *     caller sees it, is unchanged.
 *   - Arguments are validated on the host before anything is launched; a
 *     rejected call launches nothing and returns a status != FP8_OK.  Launch
 *     failures come back as FP8_ERR_CUDA.  Nothing throws across the ABI.
 *   - bfloat16 inputs are row-major with the given row stride (in elements).
 *     E4M3 codes are the OCP FP8 E4M3 ("fn") encoding, one byte each.
 *   - Matrix sizes are element counts; leading dimensions are in elements.
 *   - A size of zero rows is a valid no-op.
 */
#ifndef FP8FG_H
#define FP8FG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8_OK = 0,
    FP8_ERR_NULL = 1,        /* a required pointer is NULL */
    FP8_ERR_SHAPE = 2,       /* a size or leading dimension is invalid */
    FP8_ERR_ALIGN = 3,       /* a pointer or stride breaks the alignment rule */
    FP8_ERR_UNSUPPORTED = 4, /* valid request the library does not serve */
    FP8_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed */
    FP8_ERR_TIMEOUT = 6,     /* a kernel gave up waiting on a pipeline barrier */
    FP8_ERR_DEVICE_SHAPE = 7 /* a kernel found invalid device-side data (offsets) */
} fp8_status;

/*
 * FP8_ERR_UNSUPPORTED, in detail.  A call returns it, launching nothing, for:
 *   - sizes beyond the kernels' 32-bit tile and row walks (a dimension or a
 *     tile count of 2^31 or more), or a dispatch problem larger than the
 *     fixed scratch of fp8_moe_dispatch_quant_noalloc;
 *   - an fp8_out_t or fp8_bscale_t value the entry point does not take;
 *   - (GEMMs) a library build whose GEMM kernels were given a different
 *     register count than the one their per-warp-role register split is
 *     sized for (a build made with another CUDA compiler version): the
 *     split would stall the kernel, so it is refused.  Rebuild the library
 *     from source with the toolkit it targets (CUDA 13.0, sm_103a);
 *   - (GEMMs on CTA pairs) a device on which no cluster of two CTAs of the
 *     kernel can be resident.
 */

/* Output element type of the GEMMs. */
typedef enum { FP8_OUT_F32 = 0, FP8_OUT_BF16 = 1 } fp8_out_t;

/* Layout of the B-operand scales of fp8_gemm_blockscaled (K = inner dim). */
typedef enum {
    FP8_BSCALE_BLOCK128 = 0,   /* sb[N/128][K/128]: one scale per 128x128 block (weights) */
    FP8_BSCALE_ROW1x128 = 1,   /* sb[K/128][N]: one scale per (row n, K block), i.e. B was
                                  quantised 1x128 along K (the Wgrad GEMM, whose B is the
                                  128x1-quantised output gradient) */
    FP8_BSCALE_BLOCK128_T = 2  /* sb[K/128][N/128]: the 128x128 block grid stored transposed
                                  (the Dgrad GEMM reusing the Fprop weight scales) */
} fp8_bscale_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* fp8_status_str(fp8_status status);

/*
 * fp8_device_error: synchronises `stream`, then returns and clears the
 * library's device-side error word for the current device: FP8_ERR_TIMEOUT
 * if a GEMM kernel abandoned a barrier wait (bounded at about two seconds),
 * FP8_ERR_DEVICE_SHAPE if a grouped GEMM found non-monotone offsets,
 * FP8_OK otherwise.  FP8_ERR_CUDA if the synchronisation itself failed.
 */
fp8_status fp8_device_error(void* stream);

/*
 * fp8_selftest_wait_timeout: launches one thread that waits, with the same
 * bounded barrier wait the GEMM kernels use, on a barrier that nothing ever
 * completes; after the wait limit (about two seconds) it records
 * FP8_ERR_TIMEOUT for fp8_device_error() and returns, leaving the context
 * usable.  A check of the failure-detection path; the report has no
 * counterpart.  Asynchronous on `stream`.
 */
fp8_status fp8_selftest_wait_timeout(void* stream);

/*
 * fp8_quant_act_1x128 -- 1x128 activation quantisation (report section
 * 3.3.2, fine-grained quantization; group size 1x128).
 *   x   : bfloat16 [M][K], row stride ldx.                 (input)
 *   xq  : E4M3 codes [M][K], row stride ldq.               (output)
 *   sx  : float [K/128][M]: scale of row m, K group kb at sx[kb*M + m]. (output)
 * For each row m and group kb: amax = max |x| over the 128 elements,
 * s = fl32(amax / 448) (s = 1 when amax = 0), q = E4M3_RNE_satfinite(fl32(x / s)).
 * Requires K % 128 == 0, ldx >= K, ldq >= K, ldx % 8 == 0, ldq % 16 == 0,
 * x and xq 16-byte aligned, sx 4-byte aligned.  M >= 0.
 */
fp8_status fp8_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx,
                        uint8_t* xq, int64_t ldq, float* sx, void* stream);

/*
 * fp8_quant_act_1x128_e5m6 -- 1x128 activation quantisation to the E5M6
 * format (report section 3.3.1: a customised E5M6 format, 5-bit exponent and
 * 6-bit mantissa, for one class of activations; the grouping and scaling of
 * section 3.3.2).  Reading of what the report leaves open: sign bit, exponent
 * bias 15, exponent field 31 reserved for infinity/NaN, subnormals m * 2^-20,
 * largest finite value 65024; round to nearest with ties to the even mantissa,
 * saturating.  Scale s = fl32(amax / 65024) per group (s = 1 for an all-zero
 * group); code = E5M6(fl32(x / s)), the sign of a zero code taken from x.
 *   x   : bfloat16 [M][K], row stride ldx.                             (input)
 *   xq  : packed 12-bit codes, row m at xq + m * ldq_bytes: element k of the
 *         row occupies bits 12 k .. 12 k + 11 of the row's bytes, least
 *         significant first (3 K / 2 bytes per row).                  (output)
 *   sx  : float [K/128][M], as fp8_quant_act_1x128.                    (output)
 * Requires K % 128 == 0, ldx >= K, ldx % 8 == 0, ldq_bytes >= 3 K / 2,
 * ldq_bytes % 16 == 0, x and xq 16-byte aligned, sx 4-byte aligned.  M >= 0.
 */
fp8_status fp8_quant_act_1x128_e5m6(const void* x, int64_t M, int64_t K, int64_t ldx,
                                    uint8_t* xq, int64_t ldq_bytes, float* sx, void* stream);

/*
 * fp8_quant_act_128x1 -- 128x1 (token-wise transposed) activation quantisation
 * for the Wgrad GEMM, whose inner dimension is the token dimension M (report
 * sections 3.3.1-3.3.3; transposition moved out of the GEMM per section 3.5.2).
 *   x   : bfloat16 [M][K], row stride ldx.                 (input)
 *   xqT : E4M3 codes [K][M] (transposed, row stride M).    (output)
 *   sxT : float [M/128][K]: scale of column k, token group mb at sxT[mb*K + k]. (output)
 * Groups are 128 consecutive tokens of one column; scale and codes as above.
 * Requires M % 128 == 0, K % 64 == 0, ldx >= K, ldx % 8 == 0, x and xqT
 * 16-byte aligned, sxT 4-byte aligned.
 */
fp8_status fp8_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx,
                        uint8_t* xqT, float* sxT, void* stream);

/*
 * fp8_quant_act_dual -- fp8_quant_act_1x128 and fp8_quant_act_128x1 of the same
 * activation in one launch that reads it once (the Fprop or Dgrad operand and
 * the transposed Wgrad operand of X or dY, report sections 3.3.1-3.3.3).
 *   x        : bfloat16 [M][K], row stride ldx.                          (input)
 *   xq, sx   : as fp8_quant_act_1x128 (xq row stride ldq).               (output)
 *   xqT, sxT : as fp8_quant_act_128x1.                                   (output)
 * The outputs are bit for bit those of the two separate calls.  Requires
 * M % 128 == 0, K % 128 == 0, ldx >= K, ldx % 8 == 0, ldq >= K, ldq % 16 == 0,
 * x, xq, xqT 16-byte aligned, sx, sxT 4-byte aligned.  M >= 0.
 */
fp8_status fp8_quant_act_dual(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* xq,
                              int64_t ldq, float* sx, uint8_t* xqT, float* sxT, void* stream);

/*
 * fp8_quant_weight_128x128 -- 128x128 block weight quantisation (report
 * section 3.3.2; block size 128x128).
 *   w   : bfloat16 [K][N] (K = inner dimension of the Fprop GEMM), row stride ldw. (input)
 *   wq  : E4M3 codes [N][K] (K contiguous: the Fprop B operand), or NULL.  (output)
 *   wqT : E4M3 codes [K][N] (N contiguous: the Dgrad B operand), or NULL.  (output)
 *   sw  : float [N/128][K/128]: scale of block (nb, kb) at sw[nb*(K/128) + kb]. (output)
 * At least one of wq, wqT must be non-NULL.  Requires K % 128 == 0,
 * N % 128 == 0, ldw >= N, ldw % 8 == 0, w/wq/wqT 16-byte aligned.
 */
fp8_status fp8_quant_weight_128x128(const void* w, int64_t K, int64_t N, int64_t ldw,
                             uint8_t* wq, uint8_t* wqT, float* sw, void* stream);

/*
 * fp8_quant_fprop_operands -- both operands of one Fprop GEMM in a single
 * launch: the activation quantised 1x128 exactly as fp8_quant_act_1x128 and
 * the weight quantised 128x128 exactly as fp8_quant_weight_128x128 (report
 * section 3.3.2, fine-grained quantization; the two groupings of one GEMM).
 *   x, M, ldx, xq, ldq, sx : as fp8_quant_act_1x128 (x bfloat16 [M][K]).
 *   w, N, ldw, wq, wqT, sw : as fp8_quant_weight_128x128 (w bfloat16 [K][N]).
 *   K : the shared inner dimension, K % 128 == 0.
 * Codes and scales are bit-identical to the two single-operand calls.  M == 0
 * skips the activation (its pointers may be NULL), N == 0 the weight, and
 * K == 0 returns FP8_OK without launching.  Every other requirement is the
 * union of the two calls' requirements, checked before anything is launched.
 */
fp8_status fp8_quant_fprop_operands(const void* x, int64_t M, int64_t K, int64_t ldx,
                             uint8_t* xq, int64_t ldq, float* sx,
                             const void* w, int64_t N, int64_t ldw,
                             uint8_t* wq, uint8_t* wqT, float* sw, void* stream);

/*
 * fp8_gemm_blockscaled -- C[M][N] = sum_kb sa[m,kb] * sb(n,kb) * P_kb[m][n],
 * P_kb[m][n] = sum over k in [128 kb, 128 kb + 128) of aq[m][k] * bq[n][k]
 * (report section 3.3.2, Figure 7(b): tensor-core partial sums over each
 * 128-wide K interval, promoted to FP32 with the two scales applied).
 *   aq : E4M3 [M][K], K contiguous (row stride K).                    (input)
 *   sa : float [K/128][M]  (layout of fp8_quant_act_1x128 / 128x1).   (input)
 *   bq : E4M3 [N][K], K contiguous (row stride K).                    (input)
 *   sb : float, layout per `bmode` (fp8_bscale_t).                    (input)
 *   c  : [M][N] row stride ldc, float (FP8_OUT_F32) or bfloat16 RNE (FP8_OUT_BF16). (output)
 * Partial sums are exact-order FP32 tensor-core accumulations of one K block;
 * promotion and the cross-block sum are FP32 fused multiply-adds.
 * Requires K % 128 == 0, K > 0, N % 128 == 0, ldc >= N, ldc*elt % 16 == 0,
 * aq/bq/c 16-byte aligned, sa/sb 4-byte aligned, M >= 0.
 */
fp8_status fp8_gemm_blockscaled(const uint8_t* aq, const float* sa, const uint8_t* bq,
                         const float* sb, fp8_bscale_t bmode, int64_t M, int64_t N, int64_t K,
                         void* c, int64_t ldc, fp8_out_t out_type, void* stream);

/*
 * fp8_gemm_blockscaled_ws -- fp8_gemm_blockscaled with a split-K workspace for
 * the dense 256-column kernels (N % 256 == 0), which run on pairs of SMs.
 * When the last wave of whole 256 x 256 tiles would leave at least half of
 * the pairs idle, its tiles are cut along K into chunks computed on the idle
 * pairs; each chunk parks its FP32 partial in the workspace, and the last
 * chunk of a tile to finish adds the partials in chunk order and stores the
 * tile.  The sum of the chunks is a different FP32 rounding order than the
 * unsplit tile's (within the same error bound); it is the same for every call
 * with the same shape on the same device.
 *   workspace       : device memory, 16-byte aligned, at least
 *                     fp8_gemm_blockscaled_workspace_size() bytes, zero-filled
 *                     before its first use (each call leaves its counters zero
 *                     again).  Owned by the caller.
 *   workspace_bytes : its size.
 * Calls that share one workspace must not run concurrently (they reuse its
 * counters and partials).  Returns FP8_ERR_NULL for a NULL workspace,
 * FP8_ERR_ALIGN for a misaligned one, FP8_ERR_SHAPE for one that is too small;
 * everything else as fp8_gemm_blockscaled.
 */
fp8_status fp8_gemm_blockscaled_ws(const uint8_t* aq, const float* sa, const uint8_t* bq,
                                   const float* sb, fp8_bscale_t bmode, int64_t M, int64_t N,
                                   int64_t K, void* c, int64_t ldc, fp8_out_t out_type,
                                   void* workspace, int64_t workspace_bytes, void* stream);

/*
 * fp8_gemm_blockscaled_workspace_size -- bytes of the split-K workspace for the
 * current device (4 KB of counters + 256 KB per pair of SMs), or -1 if the
 * device cannot be queried.
 */
int64_t fp8_gemm_blockscaled_workspace_size(void);

/*
 * fp8_gemm_blockscaled_bf16a -- fp8_gemm_blockscaled with the activation
 * quantisation fused into the GEMM: A is read as bfloat16 and quantised 1x128
 * inside the kernel, on its way from the TMA copy to the tensor cores (report
 * section 3.5.2: the fusion of FP8 format conversion with TMA access).  The
 * codes and scales are those of fp8_quant_act_1x128, so C is bitwise the
 * result of fp8_quant_act_1x128 followed by fp8_gemm_blockscaled.
 *   x  : bfloat16 [M][K], row stride ldx (the activation).            (input)
 *   bq, sb, bmode : as fp8_gemm_blockscaled (FP8_BSCALE_BLOCK128 or
 *        FP8_BSCALE_BLOCK128_T).                                       (input)
 *   c  : [M][N] row stride ldc, float or bfloat16 per out_type.        (output)
 * Requires N % 256 == 0, K % 128 == 0, K > 0, ldx >= K, ldx % 8 == 0,
 * ldc >= N, ldc*elt % 16 == 0, x/bq/c 16-byte aligned, sb 4-byte aligned.
 */
fp8_status fp8_gemm_blockscaled_bf16a(const void* x, int64_t ldx, const uint8_t* bq,
                                      const float* sb, fp8_bscale_t bmode, int64_t M, int64_t N,
                                      int64_t K, void* c, int64_t ldc, fp8_out_t out_type,
                                      void* stream);

/*
 * fp8_grouped_gemm_moe_bf16a -- fp8_grouped_gemm_moe with the activation
 * quantisation fused in the same way: the expert-grouped rows x [T][K] are
 * read as bfloat16 (row stride ldx) and quantised 1x128 in the kernel; C is
 * bitwise fp8_quant_act_1x128 followed by fp8_grouped_gemm_moe.  Other
 * arguments, checks and the device-side offset validation as
 * fp8_grouped_gemm_moe; requires N % 256 == 0.
 */
fp8_status fp8_grouped_gemm_moe_bf16a(const void* x, int64_t ldx, const uint8_t* bq,
                                      const float* sb, const int32_t* offsets, int32_t E,
                                      int64_t T, int64_t N, int64_t K, void* c,
                                      fp8_out_t out_type, void* stream);

/*
 * The MXFP8 variant (power-of-two scales).  The report wishes that the
 * per-group dequantisation could be completed inside the tensor cores
 * (section 3.5.2); Blackwell's block-scaled MMA does that, but only with
 * power-of-two scales (UE8M0 exponents).  These three calls quantise with the
 * smallest power-of-two scale 2^e such that amax / 2^e <= 448 (e in
 * [-127, 127]; e = 0 for an all-zero group) and multiply with the scales
 * applied inside the tensor core, accumulating the whole K range in FP32 in
 * tensor memory.  With such scales the result is the same block-scaled
 * product as fp8_gemm_blockscaled computes; the codes differ from the amax/448
 * quantisers' (a different scale), so the variant is an alternative
 * quantisation, not a drop-in for the other calls' outputs.
 */

/*
 * fp8_quant_act_1x128_pow2 -- 1x128 activation quantisation with power-of-two
 * scales.
 *   x   : bfloat16 [M][K], row stride ldx.                             (input)
 *   xq  : E4M3 codes [M][K], row stride ldq; code = E4M3_RNE_satfinite(x / 2^e),
 *         x / 2^e exact.                                               (output)
 *   se8 : UE8M0 bytes [K/128][M]: e + 127 of row m, K group kb at se8[kb*M + m]. (output)
 * Requires K % 128 == 0, ldx >= K, ldq >= K, ldx % 8 == 0, ldq % 16 == 0,
 * x and xq 16-byte aligned.  M >= 0.
 */
fp8_status fp8_quant_act_1x128_pow2(const void* x, int64_t M, int64_t K, int64_t ldx,
                                    uint8_t* xq, int64_t ldq, uint8_t* se8, void* stream);

/*
 * fp8_quant_weight_128x128_pow2 -- 128x128 weight quantisation with
 * power-of-two scales.
 *   w   : bfloat16 [K][N], row stride ldw.                             (input)
 *   wq  : E4M3 codes [N][K] (K contiguous).                            (output)
 *   se8 : UE8M0 bytes [K/128][N]: the exponent of the block holding row n of
 *         wq, K group kb, at se8[kb*N + n] (each block's byte on its 128 rows:
 *         the per-row layout fp8_gemm_mxfp8 reads).                   (output)
 * Requires K % 128 == 0, N % 128 == 0, ldw >= N, ldw % 8 == 0, w and wq
 * 16-byte aligned.
 */
fp8_status fp8_quant_weight_128x128_pow2(const void* w, int64_t K, int64_t N, int64_t ldw,
                                         uint8_t* wq, uint8_t* se8, void* stream);

/*
 * fp8_gemm_mxfp8 -- C[M][N] = sum over k of (aq[m][k] 2^ea) (bq[n][k] 2^eb),
 * ea = sa_e8[k/128][m] - 127, eb = sb_e8[k/128][n] - 127, on the block-scaled
 * tensor-core path (tcgen05.mma kind::mxf8f6f4): each 32-element K slice of a
 * row carries its exponent into the MMA and the whole K range accumulates in
 * FP32 in tensor memory.
 *   aq    : E4M3 [M][K], K contiguous.  sa_e8: uint8 [K/128][M].       (input)
 *   bq    : E4M3 [N][K], K contiguous.  sb_e8: uint8 [K/128][N].       (input)
 *   c     : [M][N] row stride ldc, float or bfloat16 RNE per out_type. (output)
 * Requires K % 128 == 0, K > 0, N % 128 == 0, ldc >= N, ldc*elt % 16 == 0,
 * aq/bq/c 16-byte aligned, M >= 0.  Launched with programmatic stream
 * serialisation like the other GEMMs.
 */
fp8_status fp8_gemm_mxfp8(const uint8_t* aq, const uint8_t* sa_e8, const uint8_t* bq,
                          const uint8_t* sb_e8, int64_t M, int64_t N, int64_t K, void* c,
                          int64_t ldc, fp8_out_t out_type, void* stream);

/*
 * fp8_grouped_gemm_moe -- per-expert block-scaled GEMM over rows grouped by
 * expert (report section 3.4: MoE expert GEMMs; section 3.4.2: decode-time
 * batches of at most a few hundred tokens per expert are memory bound).
 *   aq      : E4M3 [T][K], rows of expert e at offsets[e] .. offsets[e+1]-1. (input)
 *   sa      : float [K/128][T].                                            (input)
 *   bq      : E4M3 [E][N][K] (each expert's weight, K contiguous).         (input)
 *   sb      : float [E][N/128][K/128].                                     (input)
 *   offsets : int32 [E+1] in DEVICE memory, offsets[0] = 0, non-decreasing,
 *             offsets[E] <= T.  Read by the kernel (no host synchronisation);
 *             invalid offsets make the kernel skip all work and raise
 *             FP8_ERR_DEVICE_SHAPE in fp8_device_error().                 (input)
 *   c       : [T][N] row stride N, float or bfloat16 per out_type.  Rows not
 *             covered by any expert are left untouched.                    (output)
 * Same per-expert arithmetic as fp8_gemm_blockscaled with FP8_BSCALE_BLOCK128.
 * Requires 1 <= E <= 65536, T >= 0, K % 128 == 0, K > 0, N % 128 == 0,
 * aq/bq/c 16-byte aligned, sa/sb/offsets 4-byte aligned.
 */
fp8_status fp8_grouped_gemm_moe(const uint8_t* aq, const float* sa, const uint8_t* bq,
                         const float* sb, const int32_t* offsets, int32_t E, int64_t T,
                         int64_t N, int64_t K, void* c, fp8_out_t out_type, void* stream);

/*
 * fp8_grouped_gemm_moe_dgrad -- the Dgrad of the grouped expert GEMM: per
 * expert e, dX_e = dY_e . W_e^T (report section 3.3.1: Dgrad in FP8 like
 * Fprop; section 3.4: MoE experts), reusing each expert's 128x128 weight
 * quantisation: the codes in the transposed orientation and the scales read
 * transposed (as FP8_BSCALE_BLOCK128_T does for the dense GEMM).
 *   aq      : E4M3 [T][K], the output gradients dY of the packed rows,
 *             quantised 1x128 along K (K = the Fprop output width).     (input)
 *   sa      : float [K/128][T].                                         (input)
 *   bq      : E4M3 [E][N][K]: per expert the wqT codes of
 *             fp8_quant_weight_128x128 (N = the Fprop inner dimension). (input)
 *   sb      : float [E][K/128][N/128]: per expert the sw scales of
 *             fp8_quant_weight_128x128, unchanged.                      (input)
 *   offsets, c, out_type, E, T: as fp8_grouped_gemm_moe (c is dX [T][N]).
 * Same checks and device-side offset validation as fp8_grouped_gemm_moe.
 */
fp8_status fp8_grouped_gemm_moe_dgrad(const uint8_t* aq, const float* sa, const uint8_t* bq,
                               const float* sb, const int32_t* offsets, int32_t E, int64_t T,
                               int64_t N, int64_t K, void* c, fp8_out_t out_type, void* stream);

/*
 * fp8_quant_act_128x1_grouped -- the 128x1 (token-wise, transposed)
 * quantisation of expert-grouped rows for the MoE Wgrad GEMM, whose
 * contraction runs over each expert's own tokens (report sections 3.3.1-3.3.3:
 * Wgrad in FP8 on 128x1 groups along the tokens; section 3.4: MoE experts).
 * Expert e's rows offsets[e] .. offsets[e+1]-1 form ceil(t_e/128) groups of
 * 128 consecutive tokens; the last group of an expert is short and is read as
 * if padded with zero rows (zero codes, no effect on its amax or the product).
 *   x       : bfloat16 [T][K], row stride ldx.                          (input)
 *   offsets : int32 [E+1] in DEVICE memory (offsets[0] = 0, non-decreasing,
 *             offsets[E] <= T; other values give unspecified results but
 *             no access outside x, xqT, sxT).                           (input)
 *   xqT     : E4M3 [K][Tp]: expert e's codes in columns pofs[e] .. pofs[e+1]-1,
 *             padding columns 0.  Columns >= pofs[E] are untouched.     (output)
 *   sxT     : float [Tp/128][K]: scale of group g (padded column 128 g), column k
 *             at sxT[g*K + k].                                          (output)
 *   pofs    : int32 [E+1] in device memory: pofs[e] = sum over e' < e of
 *             128 ceil(t_e'/128).                                       (output)
 * Requires K % 64 == 0, ldx >= K, ldx % 8 == 0, 1 <= E <= 65536,
 * Tp % 128 == 0 and Tp >= T + 127 E rounded up to 128; x, xqT 16-byte aligned,
 * sxT, offsets, pofs 4-byte aligned.
 */
fp8_status fp8_quant_act_128x1_grouped(const void* x, int64_t T, int64_t K, int64_t ldx,
                                const int32_t* offsets, int32_t E, uint8_t* xqT, float* sxT,
                                int64_t Tp, int32_t* pofs, void* stream);

/*
 * fp8_grouped_gemm_moe_wgrad -- the Wgrad of the grouped expert GEMM: per
 * expert e, dW_e[M][N] = X_e^T . dY_e, the contraction running over the
 * expert's padded token columns pofs[e] .. pofs[e+1]-1 in 128-token blocks,
 * each block's partial promoted to FP32 with the per-row A scale and the
 * per-column B scale (report section 3.3.2, Figure 7(b); section 3.3.1,
 * Wgrad in FP8).  Operands as fp8_quant_act_128x1_grouped produces them.
 *   aqT  : E4M3 [M][Tp]: the activations' transposed codes (M = the Fprop
 *          inner dimension).                                            (input)
 *   sa   : float [Tp/128][M].                                           (input)
 *   bqT  : E4M3 [N][Tp]: the output gradients' transposed codes.        (input)
 *   sb   : float [Tp/128][N].                                           (input)
 *   pofs : int32 [E+1] in device memory: multiples of 128, pofs[0] = 0,
 *          non-decreasing, pofs[E] <= Tp; invalid values make the kernel skip
 *          all work and raise FP8_ERR_DEVICE_SHAPE in fp8_device_error(). (input)
 *   c    : float [E][M][N] (FP32, the weight gradients); an expert with no
 *          tokens gets zeros.                                           (output)
 * Requires M % 128 == 0, N % 128 == 0, Tp % 128 == 0, 1 <= E <= 65536;
 * aqT, bqT, c 16-byte aligned, sa, sb, pofs 4-byte aligned.
 */
fp8_status fp8_grouped_gemm_moe_wgrad(const uint8_t* aqT, const float* sa, const uint8_t* bqT,
                               const float* sb, const int32_t* pofs, int32_t E, int64_t Tp,
                               int64_t M, int64_t N, float* c, void* stream);

/*
 * fp8_moe_dispatch_workspace_size -- bytes of device workspace
 * fp8_moe_dispatch_quant needs for T tokens and n_local local experts
 * (0 when T = 0).  *bytes is set to 0 on error.
 */
fp8_status fp8_moe_dispatch_workspace_size(int64_t T, int32_t n_local, size_t* bytes);

/*
 * fp8_moe_dispatch_quant -- MoE dispatch packing in FP8: the activation rows
 * of the tokens routed to each local expert, gathered expert by expert and
 * quantised 1x128 (report section 3.3.3: activations are dispatched to the
 * MoE experts in FP8 with the fine-grained scheme; section 3.4: expert
 * parallelism).  Produces the A operand, A scales and offsets of
 * fp8_grouped_gemm_moe.
 *   x          : bfloat16 [T][K], row stride ldx (the tokens).           (input)
 *   topk_ids   : int32 [T][topk], the experts each token is routed to
 *                (global ids; repeats within a row count once).          (input)
 *   expert_begin, n_local : the local experts are global ids
 *                expert_begin .. expert_begin + n_local - 1; local expert
 *                e = id - expert_begin; other ids are ignored.
 *   xq         : E4M3 [cap][K] (row stride K): rows offsets[e] ..
 *                offsets[e+1]-1 are the tokens routed to local expert e, in
 *                ascending token order, each quantised exactly as
 *                fp8_quant_act_1x128 quantises it.                       (output)
 *   sx         : float [K/128][cap]: scale of packed row r, K group kb at
 *                sx[kb*cap + r] (pass T = cap to fp8_grouped_gemm_moe).  (output)
 *   offsets    : int32 [n_local+1], offsets[0] = 0, offsets[n_local] = rows used. (output)
 *   token_ids  : int32 [cap]: the source token of each packed row.       (output)
 *   workspace  : device memory of fp8_moe_dispatch_workspace_size() bytes,
 *                256-byte aligned; no initialisation needed (every call
 *                overwrites what it reads).  Calls sharing a workspace must
 *                not overlap on the GPU.
 * Rows at or past offsets[n_local] (and their scales) are left untouched.
 * Placement is deterministic (no atomics on global memory).
 * Requires K % 128 == 0, K > 0, ldx >= K, ldx % 8 == 0, 1 <= topk <= 16,
 * 1 <= n_local <= 1024, cap >= T * min(topk, n_local), cap < 2^31,
 * T <= 2^27; x and xq 16-byte aligned, sx/topk_ids/offsets/token_ids 4-byte
 * aligned.  T = 0 only zeroes offsets.
 */
fp8_status fp8_moe_dispatch_quant(const void* x, int64_t T, int64_t K, int64_t ldx,
                           const int32_t* topk_ids, int32_t topk, int32_t expert_begin,
                           int32_t n_local, uint8_t* xq, float* sx, int64_t cap,
                           int32_t* offsets, int32_t* token_ids, void* workspace,
                           size_t workspace_bytes, void* stream);

/*
 * fp8_moe_dispatch_quant_noalloc -- fp8_moe_dispatch_quant without a
 * caller-provided workspace.  The report has no counterpart: this entry point
 * exists for callers that cannot hand the library device memory at the call
 * site -- C callers without a device memory pool of their own, and code that
 * must not call an allocator between its kernel launches (a device allocation
 * can synchronise the device).  The library allocates nothing here either:
 * the scratch is a fixed array in the library's device memory, one per
 * device, of 65536 int32 (256 KB).
 *   Same arguments, outputs, checks and results as fp8_moe_dispatch_quant,
 *   minus workspace and workspace_bytes.
 *   Limit: n_local * ceil(T / 64) + n_local <= 65536 (e.g. T <= 131008 tokens
 *   with 32 local experts); larger problems return FP8_ERR_UNSUPPORTED and
 *   launch nothing.
 *   Nothing needs to start at zero: every call overwrites the scratch it
 *   reads.
 *   Overlapping calls on one device (on different streams, or from different
 *   host threads without ordering) share the scratch and race; serialise them.
 *   The first call in each CUDA context looks up the scratch's device
 *   address (cudaGetSymbolAddress) with that context current and caches it,
 *   tagged with the context's id; a later call in another context of the
 *   same device (one the caller made with the driver API, or the primary
 *   context re-created after cudaDeviceReset) looks it up again.  Make the
 *   first call in a context before any stream capture begins.
 */
fp8_status fp8_moe_dispatch_quant_noalloc(const void* x, int64_t T, int64_t K, int64_t ldx,
                                   const int32_t* topk_ids, int32_t topk, int32_t expert_begin,
                                   int32_t n_local, uint8_t* xq, float* sx, int64_t cap,
                                   int32_t* offsets, int32_t* token_ids, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8FG_H */

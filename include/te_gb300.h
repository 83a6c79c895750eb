/*
 * te_gb300.h -- C ABI of the quantized linear-layer hot path on GB300 (sm_103a).
 *
 * One shared library, libte_gb300.so, holds every kernel of the path:
 *   per-tensor amax -> DelayedScaling / CurrentScaling scale update ->
 *   saturating FP8 cast / MXFP8 / NVFP4 block quantizers (row-wise and
 *   column-wise copies from one read) -> tensor-core GEMMs (tcgen05 + TMEM,
 *   TMA-fed) with the dequantization scale and bias applied in the epilogue.
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller (for example
 *    torch allocations).  No entry point allocates, frees or synchronises;
 *    work is enqueued on `stream` (a cudaStream_t passed as void*, NULL = the
 *    legacy default stream) in call order.
 *  - Matrices are row-major.  X [R, C] has its contraction dimension along C
 *    for the "row copy"; the "col copy" is the quantized transpose [C, R] with
 *    its blocks along R (the token dimension), the operand Wgrad needs.
 *  - Every GEMM computes D[m, n] = alpha * sum_k A[m, k] * B[n, k] (+ bias[n])
 *    with A [M, K] and B [N, K] both contraction-major (K contiguous).  For a
 *    linear layer Y = X W^T + b ("Introduction to FP8 training using
 *    Transformer Engine", section "Transformer Engine の使い方", te.Linear with
 *    bias=True): Fprop A = X row copy, B = W row copy; Dgrad A = dY row copy,
 *    B = W col copy; Wgrad A = dY col copy, B = X col copy ("How to Optimize
 *    Transformer-Based Models for Low-Precision Training", section
 *    "autocast モードの使用と事前量子化の比較": Fprop, Dgrad and Wgrad shapes).
 *  - Dimensions must be multiples of 16 (the tensor-core constraint stated in
 *    "Introduction to FP8 training using Transformer Engine", section
 *    "HuggingFace BERT を例にした Transformer Engine の適用", te_patch.py comment);
 *    further constraints are listed per call.  Pointers must be 16-byte aligned.
 *  - Arguments are validated on the host before anything is enqueued; a
 *    rejected call enqueues nothing and returns a non-zero te_status.  There is
 *    never a silent fallback to another precision.
 *  - Kernels that wait on the hardware (mbarrier waits in the GEMMs) give up
 *    after about two seconds, record TE_ERR_TIMEOUT in a device error word and
 *    return; te_get_last_error() reads it.
 *  - Block-scale tensors (MXFP8 E8M0, NVFP4 UE4M3) are stored in the tensor-core
 *    layout: 128-row x 4-column tiles of 512 bytes, tile-major by (row tile,
 *    column tile); inside a tile, (r, j) sits at byte (r % 32) * 16 +
 *    ((r % 128) / 32) * 4 + (j % 4).  Rows are padded to a multiple of 128 and
 *    scale columns to a multiple of 4 (MXFP8) or 16 (NVFP4); padding is written
 *    as zero by the quantizers.  te_scale_bytes() gives the size,
 *    te_scale_unswizzle() the logical [rows, cols/block] matrix.
 *  - E2M1 codes are packed two per byte, element 2i in the low nibble.
 */
#ifndef TE_GB300_H
#define TE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TE_OK = 0,
  TE_ERR_NULL = 1,        /* a required pointer is NULL */
  TE_ERR_SHAPE = 2,       /* a dimension violates the call's constraints */
  TE_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned */
  TE_ERR_DTYPE = 4,       /* dtype not accepted by this call */
  TE_ERR_UNSUPPORTED = 5, /* combination not implemented (never a fallback) */
  TE_ERR_CUDA = 6,        /* a CUDA runtime call failed (launch, memset, ...) */
  TE_ERR_TIMEOUT = 7,     /* a device-side wait gave up (reported asynchronously) */
  TE_ERR_ARG = 8          /* other invalid argument (recipe field, flag) */
} te_status;

typedef enum {
  TE_F32 = 0,
  TE_BF16 = 1,
  TE_E4M3 = 2,   /* OFP8 E4M3, saturating, max 448 */
  TE_E5M2 = 3,   /* OFP8 E5M2, saturating, max 57344 */
  TE_E2M1 = 4,   /* OCP MX FP4, max 6 */
  TE_E8M0 = 5,   /* MXFP8 block scale 2^(b-127) */
  TE_UE4M3 = 6   /* NVFP4 block scale */
} te_dtype;

/* Scaling recipe ("Introduction to FP8 training using Transformer Engine",
 * section "Transformer Engine の使い方": DelayedScaling(fp8_format=HYBRID,
 * amax_history_len=16, amax_compute_algo="max"); NeMo keys fp8_margin,
 * fp8_interval, fp8_amax_history_len, fp8_amax_compute_algo).  HYBRID is
 * {fwd_fmt = TE_E4M3, bwd_fmt = TE_E5M2}. */
typedef struct {
  te_dtype fwd_fmt;        /* TE_E4M3 or TE_E5M2: activations and weights */
  te_dtype bwd_fmt;        /* TE_E4M3 or TE_E5M2: gradients */
  int amax_history_len;    /* L >= 1 */
  int amax_compute_algo;   /* 0 = max over the history, 1 = most recent */
  int margin;              /* scale = (fmax / amax) / 2^margin, 0 <= margin <= 64 */
  int interval;            /* recompute the scale every `interval` steps, >= 1 */
} te_recipe;

enum { TE_ALGO_MAX = 0, TE_ALGO_MOST_RECENT = 1 };

/* NVFP4 quantizer flags. */
enum {
  TE_NVFP4_2D = 1u,       /* one scale per 16x16 tile (weights); copies stay transposes */
  TE_NVFP4_RHT_COL = 2u,  /* random Hadamard transform (16 points, along R) on the col copy */
  TE_NVFP4_SR = 4u        /* stochastic rounding of the E2M1 elements (gradients) */
};

/* ---- amax ---------------------------------------------------------------------
 * amax[0] = max |x| over x [rows, cols] (dtype TE_BF16 or TE_F32, NaN-free).
 * The extra per-tensor memory pass named in "How to Optimize Transformer-Based
 * Models for Low-Precision Training", section "実モデルにおける結果の解釈"
 * (NVFP4 overheads), and the input of CurrentScaling.
 * amax_rht (nullable): max |y| where y is x's column-wise view transformed by
 * the 16-point random Hadamard transform along the rows (chunks of 16 rows,
 * signs from the low 16 bits of rht_signs; see te_quantize_nvfp4), taken in the
 * same read.  Both outputs are device fp32 scalars, overwritten (not max-ed); amax
 * may be NULL when amax_rht is not (only the rotated amax, as the RHT col copy
 * needs), TE_ERR_NULL when both are.
 * rows % 16 == 0, cols % 16 == 0; rows * cols may be 0 (amax = 0). */
te_status te_amax_reduce(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols,
                         float* amax, float* amax_rht, uint32_t rht_signs, void* stream);

/* ---- scale update -------------------------------------------------------------
 * DelayedScaling bookkeeping for n_tensors tensors of one direction
 * (is_backward = 0: recipe.fwd_fmt, 1: recipe.bwd_fmt).  For tensor i, with
 * L = amax_history_len:  hist[i*L + step % L] = amax[i]; then, when
 * (step + 1) % interval == 0:  a = max(hist[i*L .. i*L+L-1]) (algo max) or
 * amax[i] (most recent); if a is finite and > 0 and the new scale
 * s = fl32(fl32(fmax / a) * 2^-margin) is finite, scale[i] = s;
 * scale_inv[i] = fl32(1 / scale[i]).  fmax = 448 (E4M3) or 57344 (E5M2).
 * A NaN amax is recorded like any other; the maximum over a window that holds
 * it is NaN, so the scale is held while it stays in the window (as for +Inf).
 * ("Introduction to FP8 training using Transformer Engine", section
 * "FP8 Training について": one scaling factor per tensor, refreshed every step.)
 * Initial state expected from the caller: hist = 0, scale = scale_inv = 1.
 * All arrays are device fp32: hist [n_tensors * L], amax/scale/scale_inv [n_tensors]. */
te_status te_scale_update(const te_recipe* recipe, int is_backward, int n_tensors, float* hist,
                          const float* amax, float* scale, float* scale_inv, int64_t step,
                          void* stream);

/* ---- per-tensor FP8 cast ---------------------------------------------------------
 * q = fmt(fl32(x * s)), round-to-nearest-even, saturating to +-fmax.
 * fmt: TE_E4M3 or TE_E5M2.  x [rows, cols] TE_BF16 or TE_F32.
 * compute_scale = 0 (DelayedScaling): s = *scale (device); amax_out (nullable)
 *   receives max|x| from the same read (fused amax).
 * compute_scale = 1 (CurrentScaling): a = max|x| is computed first into
 *   amax_out (required); s = fl32(fmax / a), or 1 when a = 0 or the quotient is
 *   not finite; `scale` is ignored (may be NULL).
 * scale_inv_out (nullable): fl32(1 / s), the dequantization factor the GEMM uses.
 * q_row [rows, cols] and q_col [cols, rows] (the transpose) are each nullable;
 * both are written from one read of x.  rows % 16 == 0, cols % 16 == 0. */
te_status te_quantize_fp8(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, te_dtype fmt,
                          const float* scale, int compute_scale, uint8_t* q_row, uint8_t* q_col,
                          float* amax_out, float* scale_inv_out, void* stream);

/* Bias gradient fused with the FP8 quantization of dY ("How to Optimize Transformer-Based
 * Models for Low-Precision Training": te.Linear(bias=True) layers; "Introduction to FP8
 * training using Transformer Engine", section "Transformer Engine の使い方"): the same as
 * te_quantize_fp8, and in the same read of x, dbias[c] = sum over rows r of x[r, c]
 * (device fp32 [cols]).  Each 64-row tile's column sums (rows in order, fp32) go to
 * `workspace` (device fp32, at least te_dbias_workspace_bytes(rows, cols) bytes, caller
 * owned, 16-byte aligned, no initial contents needed: every entry is written); a second
 * launch adds them over the tiles in a fixed order, so the result does not depend on timing.
 * dbias NULL: exactly te_quantize_fp8.  rows == 0: dbias = 0.  Errors as te_quantize_fp8,
 * plus TE_ERR_NULL (no workspace), TE_ERR_SHAPE (workspace too small), TE_ERR_ALIGN. */
size_t te_dbias_workspace_bytes(int64_t rows, int64_t cols);
te_status te_quantize_fp8_dbias(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, te_dtype fmt,
                                const float* scale, int compute_scale, uint8_t* q_row, uint8_t* q_col,
                                float* amax_out, float* scale_inv_out, float* dbias, float* workspace,
                                size_t workspace_bytes, void* stream);

/* ---- MXFP8 ----------------------------------------------------------------------
 * Blocks of 32 consecutive elements along the contraction dimension (OCP MX
 * v1.0): E = clamp(floor(log2 a_b) - 8, -127, 127) (a_b = block amax; a_b = 0
 * gives -127), scale byte E + 127 (E8M0), q = E4M3(fl32(x * 2^-E)).
 * Row copy: q_row [rows, cols], s_row scales of [rows, cols/32];
 * col copy: q_col [cols, rows], s_col scales of [cols, rows/32].
 * Each (q, s) pair is nullable as a pair.  rows % 32 == 0 if the col copy is
 * requested, cols % 32 == 0 if the row copy is requested, both % 16. */
te_status te_quantize_mxfp8(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols,
                            uint8_t* q_row, uint8_t* s_row, uint8_t* q_col, uint8_t* s_col,
                            void* stream);

/* ---- NVFP4 ------------------------------------------------------------------------
 * Per copy: S_enc = fl32(2688 / A) (A = tensor amax of that copy's view; 1 when
 * A = 0 or the quotient overflows), S_dec = fl32(1 / S_enc).  Per block of 16
 * along the contraction (or 16x16 tile with TE_NVFP4_2D):
 *   s_b = UE4M3(fl32(fl32(a_b / 6) * S_enc));  r = fl32(S_enc / s_b) (0 if s_b = 0);
 *   q = E2M1(fl32(x * r))  -- round-to-nearest-even, or stochastic with TE_NVFP4_SR.
 * ("How to Optimize Transformer-Based Models for Low-Precision Training",
 * section "実モデルにおける結果の解釈": random Hadamard transform on the Wgrad
 * inputs, stochastic rounding of gradients, 2D block scaling of weights, an
 * extra pass for the per-tensor amax.)
 * amax: device scalar A of x (from te_amax_reduce), required if the row copy or
 *   an unrotated col copy is requested.  amax_rht: A of the rotated col view,
 *   required with TE_NVFP4_RHT_COL.
 * RHT (col copy only): every chunk of 16 rows of a column is replaced by
 *   (1/4) H16 D x, H16 the Sylvester Hadamard matrix, D = diag(-1 where bit j of
 *   rht_signs is set); fp32 evaluation: sign flip, butterflies h = 1, 2, 4, 8
 *   ((u, v) -> (u + v, u - v)), then * 0.25.
 * SR: with a = |v| between E2M1 neighbours lo <= a < hi and frac = (a - lo) / (hi - lo),
 *   the magnitude rounds up iff R + floor(frac * 2^16) >= 2^16 (a >= 6 saturates; the
 *   sign is kept).  Element g (row-major index inside the copy) belongs to the group
 *   of four g / 4, which reads word w = word (g / 4) % 4 of Philox4x32-10(counter =
 *   (g / 16, copy_id, offset_lo, offset_hi), key = (seed_lo, seed_hi)), copy_id 0 for
 *   the row copy and 1 for the col copy; with P = (w[23:16] << 8) | w[7:0] and
 *   Q = (w[31:24] << 8) | w[15:8], positions 0..3 of the group take R = P,
 *   bitrev16(P), Q, bitrev16(Q) (the bit split of the hardware stochastic-rounding
 *   conversion, which rounds four values per instruction).
 * Outputs: q_row [rows, cols/2] bytes, s_row, gdec_row (device fp32 S_dec);
 *   q_col [cols, rows/2], s_col, gdec_col.  Each triple is nullable as a unit.
 * cols % 32 == 0 if the row copy is requested, rows % 32 == 0 if the col copy is
 * (the packed copies' rows must be whole 16-byte units, as the GEMM's K % 32);
 * TE_NVFP4_2D excludes TE_NVFP4_RHT_COL. */
te_status te_quantize_nvfp4(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols,
                            uint32_t flags, uint32_t rht_signs, uint64_t seed, uint64_t offset,
                            const float* amax, const float* amax_rht,
                            uint8_t* q_row, uint8_t* s_row, float* gdec_row,
                            uint8_t* q_col, uint8_t* s_col, float* gdec_col, void* stream);

/* te_quantize_fp8_dbias without a caller workspace.  The paper has no counterpart: this
 * exists for callers that cannot allocate device memory where they quantize dY -- code
 * running while a memory pool is locked or sized ahead of time, or a host runtime that
 * owns every allocation and passes only the tensors to be computed on.  The 64-row-tile
 * partial sums go to a fixed 4 MiB array inside the library (one per GPU that loads the
 * library, kept until the process exits), so ceil(rows / 64) * cols may be at most
 * 1,048,576 (e.g. 15872 x 4096); larger requests return TE_ERR_SHAPE before anything is
 * enqueued.  Arguments, outputs and other errors as te_quantize_fp8_dbias.  Nothing in
 * the array has to start at zero (each call writes every partial sum it reads), but
 * every call shares it: calls that can overlap on the GPU (other streams, other host
 * threads on the same device) race and must be ordered by the caller.  The first call
 * on a device looks up the array's device address (cudaGetSymbolAddress, with that
 * device current); make that first call before any stream capture.  The address is
 * kept for the life of the process, so a device that the library has used must not be
 * reset (cudaDeviceReset) while the library stays loaded.  Argument checks run before
 * that lookup.  No device memory is allocated or freed by this call. */
te_status te_quantize_fp8_dbias_noalloc(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, te_dtype fmt,
                                        const float* scale, int compute_scale, uint8_t* q_row, uint8_t* q_col,
                                        float* amax_out, float* scale_inv_out, float* dbias, void* stream);

/* LayerNorm fused with the FP8 cast of its output: the step before the QKV and MLP-up
 * Fprop (te.LayerNorm / the fused LayerNorm kernels of "Introduction to FP8 training
 * using Transformer Engine").  x bf16 [rows, cols] (cols % 16 == 0, cols <= 8192);
 * gamma, beta device fp32 [cols] (16-byte aligned).  Per row: mu = mean, var = biased
 * variance (fp32, fixed summation order), rsigma = 1 / sqrt(var + eps);
 * y = ((x - mu) * rsigma) * gamma + beta in fp32, rounded to bf16 -- the LN output,
 * written to ln_out (bf16 [rows, cols], nullable) -- and that bf16 value is cast to FP8
 * as te_quantize_fp8 would cast it: q_row = sat(fl32(y * scale[0])) (fmt E4M3 / E5M2,
 * DelayedScaling's scale from the history).  mu, rsigma (device fp32 [rows], nullable)
 * are kept for the backward pass; amax_out (nullable) = max |y| over the bf16 outputs;
 * scale_inv_out (nullable) = 1 / scale.  One read of x from HBM per row.  (The col copy
 * for Wgrad comes from te_quantize_fp8 on ln_out.) */
te_status te_layernorm_fp8(const void* x, te_dtype in_dtype, int64_t rows, int64_t cols, const float* gamma,
                           const float* beta, float eps, te_dtype fmt, const float* scale, uint8_t* q_row,
                           void* ln_out, float* mu, float* rsigma, float* amax_out, float* scale_inv_out,
                           void* stream);

/* ---- GEMMs ----------------------------------------------------------------------
 * Common: A [M, K], B [N, K] contraction-major; D [M, N] row-major of out_dtype
 * (TE_BF16, round-to-nearest-even, or TE_F32); bias (nullable) device fp32 [N];
 * fp32 accumulation in tensor memory; epilogue D = alpha * acc + bias.
 * accumulate = 1 (out_dtype TE_F32 only, else TE_ERR_DTYPE): D += alpha * acc + bias,
 * the Wgrad form that adds into an fp32 main gradient (the pages' fp8_wgrad /
 * weight-gradient path of "Introduction to FP8 training using Transformer Engine",
 * NeMo keys); every element of D is read, added to in fp32 and written exactly once
 * per call (a TMA reduce-add of the tile), so the result does not depend on timing.
 * M, N, K multiples of 16 (K of 32 for NVFP4).  Timing of the GEMM alone is the
 * pages' "pre-quantized" mode; quantize + GEMM is "autocast" mode. */

/* Operand storage order for te_gemm_bf16. */
typedef enum {
  TE_K_MAJOR = 0,  /* A stored [M, K] / B stored [N, K] (contraction contiguous) */
  TE_MN_MAJOR = 1  /* A stored [K, M] / B stored [K, N] (the non-contracted index contiguous) */
} te_layout;

/* BF16 x BF16 (kind::f16), alpha = 1.  Each operand may be stored either way, so
 * Dgrad (dX = dY W: B = W read MN-major) and Wgrad (dW = dY^T X: both operands
 * MN-major) need no transposed copies, as a BF16 layer has none. */
te_status te_gemm_bf16(const void* A, te_layout a_layout, const void* B, te_layout b_layout, const float* bias,
                       void* D, te_dtype out_dtype, int accumulate, int64_t M, int64_t N, int64_t K, void* stream);

/* Per-tensor scaled FP8 (kind::f8f6f4): fa, fb in {TE_E4M3, TE_E5M2};
 * alpha = a_scale_inv[0] * b_scale_inv[0] (device fp32 scalars). */
te_status te_gemm_fp8(const uint8_t* A, te_dtype fa, const uint8_t* B, te_dtype fb,
                      const float* a_scale_inv, const float* b_scale_inv, const float* bias, void* D,
                      te_dtype out_dtype, int accumulate, int64_t M, int64_t N, int64_t K, void* stream);

/* MXFP8 (kind::mxf8f6f4, block 32, E8M0 scales in the tensor-core layout), alpha = 1.
 * sA: scales of A [M, K/32]; sB: scales of B [N, K/32]; K % 32 == 0. */
te_status te_gemm_mxfp8(const uint8_t* A, te_dtype fa, const uint8_t* sA, const uint8_t* B, te_dtype fb,
                        const uint8_t* sB, const float* bias, void* D, te_dtype out_dtype, int accumulate,
                        int64_t M, int64_t N, int64_t K, void* stream);

/* NVFP4 (kind::mxf4nvf4, block 16, UE4M3 scales in the tensor-core layout);
 * A, B packed E2M1 [M, K/2], [N, K/2]; alpha = gA[0] * gB[0] (the copies' S_dec). */
te_status te_gemm_nvfp4(const uint8_t* A, const uint8_t* sA, const float* gA, const uint8_t* B,
                        const uint8_t* sB, const float* gB, const float* bias, void* D,
                        te_dtype out_dtype, int accumulate, int64_t M, int64_t N, int64_t K, void* stream);

/* ---- host helpers ------------------------------------------------------------------ */

/* Bytes of the block-scale tensor of a quantized copy with `rows` rows of `cols`
 * elements: scale_fmt TE_E8M0 (MXFP8, block 32) or TE_UE4M3 (NVFP4, block 16).
 * Returns 0 for invalid arguments. */
size_t te_scale_bytes(te_dtype scale_fmt, int64_t rows, int64_t cols);

/* Host-side: copy the tensor-core-layout scales `swizzled` (host memory,
 * te_scale_bytes long) into the logical row-major [rows, cols/block] matrix. */
te_status te_scale_unswizzle(te_dtype scale_fmt, int64_t rows, int64_t cols, const uint8_t* swizzled,
                             uint8_t* logical);

/* Human-readable name of a status. */
const char* te_status_str(te_status s);

/* Synchronises the current device, then returns and clears the first error
 * recorded by a kernel (TE_ERR_TIMEOUT) or by the CUDA runtime (TE_ERR_CUDA). */
te_status te_get_last_error(void);

/* Self-test of the device-side failure detection: launches one warp that waits on
 * a barrier nothing will complete; the bounded wait gives up after ~10 ms and the
 * kernel returns, leaving TE_ERR_TIMEOUT for the next te_get_last_error().  The
 * context stays usable (no trap, no fault). */
te_status te_selftest_wait_timeout(void* stream);

/* Number of kernels launched by this library since load (a counter the host
 * increments at every launch; for accounting in benchmarks). */
uint64_t te_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* TE_GB300_H */

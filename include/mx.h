/*
 * mx.h -- C ABI of the GB300 (sm_103a) MX block-scaled / FP16 GEMM library
 * (libmx_gb300.so).
 *
 * Three operations, all launched asynchronously on the caller's CUDA stream:
 *
 *   mx_quantize  fp32 matrix -> MX tensor (E4M3, E5M2 or E2M1 data plane plus
 *                a UE8M0 scale plane, one scale per 32 consecutive K elements)
 *   mx_gemm      C = A * B on two MX tensors, fp32 accumulation, dequantize
 *                inside the tensor-core matmul, fp32 or bf16 C
 *   gemm_f16     C = A * B on row-major fp16 or bf16 matrices, fp32
 *                accumulation, fp32 C
 *   *_fused      the same products with bias and GELU applied to the fp32
 *                accumulator in the epilogue, and mx_gemm_fused_quantize,
 *                which also quantizes C to an MX tensor for the next layer
 *
 * Where these come from.  The quantized tensor as one object holding a data
 * plane and a scale plane, the scale format ("FP8 E8M0") and the block of 32
 * along the innermost dimension are the WWDC26 session 330 pages ("Metal
 * tensors ... / Optimize custom ML ops with Metal tensors"), chapters
 * "Multi-plane tensors" (4:23) and "Quantized matrix multiplication" (5:17),
 * and the listings at 4:48 (scale plane with block factors {32, 1}) and 7:19
 * (matmul of two quantized tensors with no transposes, dequantization done
 * by the matmul).  FP16 matmul with fp32 accumulation is the "Passo 6" step
 * of the dicastech tutorial "Treinar LLM em Swift: multiplicacao de matrizes
 * do Gflop/s ao Tflop/s".  The element and scale encodings and the rule
 * X = 2^(floor(log2 amax) - emax) follow the OCP Microscaling (MX) v1.0
 * specification.
 *
 * Memory.  Every pointer argument except those of mx_scales_to_rowmajor is a
 * device pointer owned by the caller; the library never allocates, frees or
 * synchronizes on these calls (mx_last_error is the one call that
 * synchronizes).  Inputs are only read; outputs are written in full.
 *
 * Errors.  Argument, shape and alignment checks run on the host before
 * anything is launched and return a status without touching the GPU.  A
 * launch failure returns MX_ERR_CUDA.  Every wait inside a kernel is bounded;
 * a wait that runs out records MX_ERR_TIMEOUT in a device status word, the
 * kernel returns cleanly, and mx_last_error reports it.
 */
#ifndef MX_GB300_H
#define MX_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum mx_status {
  MX_OK = 0,
  MX_ERR_INVALID_ARG = 1, /* null pointer, unknown enum value             */
  MX_ERR_SHAPE = 2,       /* sizes or leading dimensions not supported     */
  MX_ERR_ALIGN = 3,       /* pointer or stride not 16-byte aligned         */
  MX_ERR_UNSUPPORTED = 4, /* no device of compute capability 10.3          */
  MX_ERR_CUDA = 5,        /* a CUDA runtime or driver call failed          */
  MX_ERR_TIMEOUT = 6      /* a kernel gave up on a bounded wait            */
} mx_status;

/* Element format of an MX data plane. */
typedef enum mx_format {
  MX_FMT_E4M3 = 1, /* MXFP8: 1 sign, 4 exponent (bias 7), 3 mantissa bits;
                      one code per byte; no infinity; max 448            */
  MX_FMT_E2M1 = 2, /* MXFP4: 1 sign, 2 exponent (bias 1), 1 mantissa bit;
                      two codes per byte, the element with even k in the
                      low nibble; max 6                                   */
  MX_FMT_E5M2 = 3, /* MXFP8 with a wider range: 1 sign, 5 exponent (bias
                      15), 2 mantissa bits; one code per byte; max 57344;
                      0x7C / 0xFC are +-infinity (mx_quantize never writes
                      them, mx_gemm propagates them), 0x7D-0x7F NaN.  The
                      RIGEL summary, Main findings section 3, names E5M2
                      beside E4M3 and notes that it has infinities.       */
  /* Integer elements (WWDC26 session 330, "Quantized data types": 8-, 4- and
     2-bit integers under the same E8M0 block scales): two's complement, an
     element's value is q * X.  mx_quantize uses emax = bits - 2 (the OCP
     MXINT8 rule for int8) and rounds to the nearest integer, ties to even,
     saturating.  The tensor cores have no block-scaled integer kind:
     integer tensors are the B operand of gemm_dequant; mx_gemm and its
     variants reject them (MX_ERR_INVALID_ARG).                            */
  MX_FMT_INT8 = 4, /* one code per byte, -128..127                          */
  MX_FMT_INT4 = 5, /* two codes per byte, even k in the low nibble, -8..7   */
  MX_FMT_INT2 = 6  /* four codes per byte, element k at bits 2*(k%4), -2..1 */
} mx_format;

/* Element type of a plain matrix. */
typedef enum mx_dtype { MX_DT_F32 = 0, MX_DT_BF16 = 1, MX_DT_F16 = 2 } mx_dtype;

/* Activation of a fused epilogue. */
typedef enum mx_activation {
  MX_ACT_NONE = 0,
  MX_ACT_GELU = 1,      /* GELU(x) = x * Phi(x), Phi the standard normal CDF  */
  MX_ACT_GELU_TANH = 2  /* its tanh approximation:
                           0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))   */
} mx_activation;

/* Orientation of mx_quantize's fp32 source. */
typedef enum mx_src_layout {
  MX_SRC_K_CONTIGUOUS = 0, /* source is outer x K row-major (the A operand)   */
  MX_SRC_K_STRIDED = 1     /* source is K x outer row-major (a row-major K x N
                              B operand); blocks of 32 still run along K     */
} mx_src_layout;

/*
 * An MX tensor: the quantized form of an outer x K matrix whose K axis is the
 * contraction axis (A: outer = M; B: outer = N).
 *
 *   data    device, outer x K codes, K contiguous, rows packed back to back:
 *           mx_data_bytes(fmt, outer, K) bytes; 16-byte aligned.
 *   scales  device, UE8M0 codes (value 2^(c-127), 0xFF = NaN) in the
 *           tensor-core scale-factor layout: the scale matrix, padded to a
 *           multiple of 128 rows and of 4 blocks, is cut into atoms of 128 rows
 *           x 4 blocks (128 K elements) of 512 contiguous bytes; the scale of
 *           (row r, block j) is byte 16*(r%32) + 4*((r%128)/32) + (j%4) of atom
 *           (r/128) * ceil(K/128) + j/4.  mx_scale_bytes(outer, K) bytes;
 *           16-byte aligned.  Padding bytes must not be 0xFF (mx_quantize
 *           writes 0 there).
 *   fmt     mx_format
 *   outer   rows (M for A, N for B), >= 0
 *   K       contraction length, a multiple of 32, >= 0
 */
typedef struct mx_tensor {
  void* data;
  uint8_t* scales;
  int32_t fmt;
  int64_t outer;
  int64_t K;
} mx_tensor;

/* Bytes of the data plane: outer*K (E4M3, E5M2, int8), outer*K/2 (E2M1,
 * int4) or outer*K/4 (int2); 0 on bad arguments. */
size_t mx_data_bytes(int32_t fmt, int64_t outer, int64_t K);

/* Bytes of the scale plane: ceil(outer/128) * ceil(K/128) * 512; 0 on bad
 * arguments. */
size_t mx_scale_bytes(int64_t outer, int64_t K);

/*
 * mx_quantize -- OCP MX quantization of an fp32 matrix into out (the planes
 * must already be allocated by the caller at the sizes above).
 *
 * For every row r of out and every block j of 32 consecutive K elements:
 *   amax = max |x| over the block; e = floor(log2(amax)) from the fp32
 *   exponent; X = 2^clamp(e - emax, -127, 127) with emax = 8 (E4M3), 15
 *   (E5M2), 2 (E2M1) or bits - 2 (the integer formats); the scale code is
 *   log2(X) + 127; each element is
 *   x / X rounded to nearest-even and saturated to the format's largest
 *   finite value (for E5M2 too: a block's own maximum, up to 1.99 * 2^15
 *   after scaling, becomes 57344, never an infinity).
 *   An all-zero block gets scale code 0; a block holding a NaN or an
 *   infinity gets scale code 0xFF (its element codes are then unspecified).
 *
 *   src         device fp32; element (r, k) at src[r*ld + k]
 *               (MX_SRC_K_CONTIGUOUS) or src[k*ld + r] (MX_SRC_K_STRIDED)
 *   ld          leading dimension in elements; ld >= K (K_CONTIGUOUS) or
 *               ld >= outer (K_STRIDED); a multiple of 4
 *   src_layout  mx_src_layout
 *   out         fmt, outer, K, data and scales as described above
 *   stream      cudaStream_t (NULL: the legacy default stream)
 * Returns MX_OK, or an error status before any launch.
 */
mx_status mx_quantize(const float* src, int64_t ld, int32_t src_layout,
                      const mx_tensor* out, void* stream);

/*
 * mx_gemm -- C = A * B^T over the MX tensors A (M x K) and B (N x K), i.e. the
 * product of the M x K matrix A and the K x N matrix that B was quantized
 * from, with fp32 accumulation:
 *   C[i][j] = sum_k (a_ik * Xa_i,k/32) * (b_jk * Xb_j,k/32).
 *
 *   A, B     MX tensors of the same K (A->outer = M, B->outer = N).  Their
 *            formats may differ: any two of E4M3, E5M2 and E2M1.  A pair
 *            of E2M1 tensors runs at the FP4 tensor rate; every other pair
 *            runs at the FP8 rate, and a pair mixing E2M1 with an 8-bit
 *            format needs K a multiple of 128 and the E2M1 data plane
 *            32-byte aligned (MX_ERR_SHAPE / MX_ERR_ALIGN otherwise).
 *   C        device, M x N row-major, element type c_dtype (MX_DT_F32 or
 *            MX_DT_BF16, rounded to nearest-even); 16-byte aligned
 *   ldc      leading dimension of C in elements, >= N; ldc * element size
 *            a multiple of 16 bytes
 *   stream   cudaStream_t
 * M, N >= 0 and K >= 0 (K a multiple of 32).  K = 0 writes C = 0.
 */
mx_status mx_gemm(const mx_tensor* A, const mx_tensor* B, void* C,
                  int32_t c_dtype, int64_t ldc, void* stream);

/*
 * gemm_f16 -- C = A * B with A (M x K) and B (K x N) row-major fp16 or bf16,
 * fp32 accumulation, fp32 C (M x N row-major).
 *
 *   ab_dtype  MX_DT_F16 or MX_DT_BF16 (both operands)
 *   lda, ldb  leading dimensions in elements (lda >= K, ldb >= N), multiples
 *             of 8; A and B 16-byte aligned
 *   ldc       >= N, a multiple of 4; C 16-byte aligned
 * K = 0 writes C = 0.
 */
mx_status gemm_f16(const void* A, const void* B, float* C, int32_t ab_dtype,
                   int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                   int64_t ldc, void* stream);

/*
 * Fused epilogue -- the GEMM + bias + GELU kernel of the RIGEL summary (Main
 * findings section 4: fusing the epilogue in registers saves the O(n^2)
 * round trip of C through memory).  Each element of the fp32 accumulator
 * becomes
 *   y[i][j] = act(acc[i][j] + bias[j])
 * in fp32 before C is stored.
 *
 *   bias  device, N fp32 values (bias[j] is added to column j), 16-byte
 *         aligned; NULL: no bias
 *   act   mx_activation
 * A NULL mx_epilogue pointer means no bias and MX_ACT_NONE.
 */
typedef struct mx_epilogue {
  const float* bias;
  int32_t act;
} mx_epilogue;

/* mx_gemm with the fused epilogue.  K = 0 is rejected (MX_ERR_SHAPE) when
 * the epilogue does anything; other arguments as for mx_gemm. */
mx_status mx_gemm_fused(const mx_tensor* A, const mx_tensor* B,
                        const mx_epilogue* epi, void* C, int32_t c_dtype,
                        int64_t ldc, void* stream);

/*
 * mx_gemm_fused_quantize -- y = act(A * B + bias) as above, then quantized
 * in the epilogue into the MX tensor C (C->outer = M, C->K = N: blocks of 32
 * consecutive columns of y share a scale, so C is ready to be the A operand
 * of a next product whose contraction runs over those N columns).  The
 * result is what mx_quantize (MX_SRC_K_CONTIGUOUS) would make of the fp32
 * output of mx_gemm_fused, without the fp32 round trip through memory.
 *
 *   C       any mx_format; N a multiple of 32; its planes must not overlap
 *           A's or B's
 * K > 0 is required (MX_ERR_SHAPE otherwise).
 */
mx_status mx_gemm_fused_quantize(const mx_tensor* A, const mx_tensor* B,
                                 const mx_epilogue* epi, const mx_tensor* C,
                                 void* stream);

/* gemm_f16 with the fused epilogue (fp32 C); K = 0 is rejected when the
 * epilogue does anything. */
mx_status gemm_f16_fused(const void* A, const void* B, const mx_epilogue* epi,
                         float* C, int32_t ab_dtype, int64_t M, int64_t N,
                         int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                         void* stream);

/*
 * gemm_dequant -- C = A * dequant(B)^T: a row-major fp16 / bf16 A (M x K)
 * times an MX tensor B (N x K) of any mx_format, with fp32 accumulation.
 * WWDC26 session 330, "Quantized matrix multiplication": a quantized format
 * the matmul cannot take directly is loaded in chunks, dequantized to f16 in
 * threadgroup memory and multiplied.  Here the CTA pair dequantizes B's codes
 * and scales into shared memory as a_dtype values and runs the 16-bit tensor
 * cores; weight-only quantization (int4 / int2 / E2M1 weights, 16-bit
 * activations) is the intended use.  Up to 128 rows of A (decoding a few
 * tokens) a second kernel takes the product: B's 128-row blocks are the MMA's
 * rows, dequantized into tensor memory 256 K at a time, A's rows its columns;
 * when the blocks are fewer than the SMs, each block's K range is split over
 * a thread-block cluster of up to 8 CTAs whose partial sums are added in a
 * fixed order on chip (no workspace, same bits every run).  A single row of
 * a bf16 A with 4- or 2-bit codes (int4, int2, E2M1: decoding one token)
 * takes a third kernel that streams B once on the CUDA cores: each lane
 * dequantizes whole 32-element blocks to the same bf16 values and sums
 * their products with A in fp32 (no workspace, same bits every run).
 *
 *   A        device, M x K, row-major, element type a_dtype (MX_DT_F16 or
 *            MX_DT_BF16); lda >= K, a multiple of 8; 16-byte aligned
 *   B        any format; K a multiple of 64
 *   epi      fused epilogue (NULL: none), as for mx_gemm_fused
 *   C        device, M x N row-major, c_dtype MX_DT_F32 or MX_DT_BF16;
 *            ldc >= N, ldc * element size a multiple of 16 bytes
 * A dequantized element q * X must lie in a_dtype's range to be exact
 * (bf16 holds every code of every format for scales 2^-120 .. 2^120; f16
 * only values up to 65504).
 */
mx_status gemm_dequant(const void* A, int32_t a_dtype, int64_t M, int64_t lda,
                       const mx_tensor* B, const mx_epilogue* epi, void* C,
                       int32_t c_dtype, int64_t ldc, void* stream);

/* gemm_dequant with a K-split: when the output tiles leave SMs idle (more
 * than 128 rows of A but few tiles), each tile's K range is split into parts
 * that run on those SMs, each writing an fp32 partial tile to the
 * workspace; a second kernel adds the parts in a fixed order, applies the
 * epilogue and writes C.  workspace: device, 16-byte aligned, at least
 * gemm_dequant_workspace_bytes(M, N, K) bytes (0: the problem is not split
 * this way -- always so for M <= 128, whose kernel splits K inside clusters
 * and ignores the workspace; NULL or smaller: the call runs unsplit). */
size_t gemm_dequant_workspace_bytes(int64_t M, int64_t N, int64_t K);
mx_status gemm_dequant_splitk(const void* A, int32_t a_dtype, int64_t M,
                              int64_t lda, const mx_tensor* B,
                              const mx_epilogue* epi, void* C, int32_t c_dtype,
                              int64_t ldc, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * flash_attention -- O = softmax(Q K^T * scale) V for BH independent heads,
 * in one kernel: the scores and probabilities stay on the SM (WWDC26
 * session 330, "Building advanced ops": Q x K, a row-max reduction, the
 * exponentials and the product with V fused, the probabilities handed to the
 * second matmul without a round trip through memory -- FlashAttention).
 *
 *   Q        device, BH x Lq x d, row-major, dtype (MX_DT_F16 / MX_DT_BF16)
 *   K, V     device, BH x Lk x d, row-major, dtype
 *   O        device, BH x Lq x d, row-major, o_dtype (MX_DT_F32, MX_DT_BF16
 *            or MX_DT_F16); every pointer 16-byte aligned
 *   d        64 or 128; Lk >= 1 when Lq >= 1; BH <= 65535
 *   scale    multiplies Q K^T (commonly 1/sqrt(d)); finite
 * The scores accumulate in fp32; the probabilities are rounded to dtype
 * before the product with V and the row sums add them in fp32, so each
 * output row is a combination of V's rows whose weights differ from the
 * exact softmax by at most that rounding (relative 2^-8 for bf16, 2^-11 for
 * f16).  No mask.
 */
mx_status flash_attention(const void* Q, const void* K, const void* V, void* O,
                          int32_t dtype, int32_t o_dtype, int64_t BH, int64_t Lq,
                          int64_t Lk, int64_t d, float scale, void* stream);

/*
 * flash_attention_splitkv -- flash_attention with the key axis split where
 * SMs would otherwise idle.  A CTA computes one (head, 256 queries) unit.
 * The units of a last, partial wave (all units, when there are fewer units
 * than SMs, as in decoding with few queries and a long context) are each cut
 * into up to 16 ranges of key blocks (at least two blocks each).  Each range
 * writes its un-normalised output rows with their reference point m and row
 * sum l into the workspace.  A second kernel merges the ranges in a fixed
 * order as sum_p 2^(m_p - M) O_p / sum_p 2^(m_p - M) l_p, where M = max_p m_p.
 * This is the exact identity behind the online softmax, so results stay
 * within the flash_attention bound; they can differ from the unsplit call
 * in the last bits.
 *
 *   workspace        device, 16-byte aligned, caller-owned scratch of at least
 *                    flash_attention_workspace_bytes() bytes; contents on
 *                    entry do not matter and are garbage after.  NULL or a
 *                    smaller size: the call runs unsplit.
 *   other arguments  as for flash_attention.
 * flash_attention_workspace_bytes returns 0 when nothing would be split (the
 * units fill whole waves, or Lk < 256), on bad arguments, or without a
 * compute capability 10.3 device.  The size depends on the device's SM count.
 */
size_t flash_attention_workspace_bytes(int64_t BH, int64_t Lq, int64_t Lk, int64_t d);
mx_status flash_attention_splitkv(const void* Q, const void* K, const void* V, void* O,
                                  int32_t dtype, int32_t o_dtype, int64_t BH, int64_t Lq,
                                  int64_t Lk, int64_t d, float scale, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * K-split variants.  When a problem's tiles leave clusters of SMs idle (a last,
 * partial wave of tiles, or fewer tiles than cluster slots), these calls
 * split the affected tiles along K across the idle clusters, inside the one
 * GEMM launch: each part writes its fp32 partial tile into the workspace and
 * counts itself on the tile's counter there; the part that completes the
 * count adds all the tile's parts in part order (the same order whichever
 * part finishes last, so results do not depend on timing) and writes C.  The
 * sum is grouped differently from the unsplit call, so the two can differ in
 * the last bits; both are within the same accumulation bound.
 *
 *   workspace        device, 16-byte aligned, caller-owned scratch of at
 *                    least *_workspace_bytes() bytes for the problem: the
 *                    partial tiles, then one 8-byte counter per split tile
 *                    and CTA.  Its contents on entry do not matter: a counter
 *                    word counts only arrivals tagged with this launch's
 *                    48-bit tag (a stale word matches it with probability
 *                    2^-48), and the completing arrival sets it to zero, so a
 *                    call replayed from a CUDA graph (same tag) starts from
 *                    zero too.  Two calls that share a workspace must not
 *                    run at the same time.
 *                    NULL or a smaller size: the call runs unsplit.
 *   other arguments  as for mx_gemm / gemm_f16.
 * *_workspace_bytes returns 0 when the problem is not split (or on bad
 * arguments, or without a compute capability 10.3 device).
 */
/* fmt: the element format of both operands; for operands of different
 * formats pass MX_FMT_E4M3. */
size_t mx_gemm_workspace_bytes(int32_t fmt, int64_t M, int64_t N, int64_t K);
mx_status mx_gemm_splitk(const mx_tensor* A, const mx_tensor* B, void* C,
                         int32_t c_dtype, int64_t ldc, void* workspace,
                         size_t workspace_bytes, void* stream);
size_t gemm_f16_workspace_bytes(int64_t M, int64_t N, int64_t K);
mx_status gemm_f16_splitk(const void* A, const void* B, float* C,
                          int32_t ab_dtype, int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, int64_t ldc, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * mx_gemm_splitk_noalloc -- mx_gemm_splitk for callers that cannot allocate
 * device memory: the split's scratch comes from a fixed 24 MiB array inside
 * the library instead of a caller-provided workspace.  The pages have no
 * counterpart to this call.
 *
 * Who needs it: code that sees only the operand and result pointers (an
 * operator or plugin interface with no workspace argument) and processes
 * whose device memory is reserved in advance by a framework's caching
 * allocator or a fixed budget, where a library cudaMalloc would fail or
 * escape the allocator's accounting.  This call makes no allocation at all.
 *
 *   A, B, C, c_dtype, ldc, stream   as for mx_gemm.
 * Returns MX_ERR_SHAPE when the problem's split would need more than the
 * 24 MiB (mx_gemm_workspace_bytes() > 24 MiB; not reachable on a 152-SM
 * GB300, where the split needs at most about 10 MiB).
 *
 * The array is shared by every call in the process: two calls whose
 * executions overlap on the GPU (different streams, or different host
 * threads) race on it and give wrong results; serialize them.  Each GPU on
 * which the library's module has been loaded keeps the 24 MiB until the
 * process exits.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) and caches it for the device's current
 * context; make that first call before any stream capture on that device.
 * After a device reset (cudaDeviceReset) the next call looks the address up
 * again, so it too must come before any capture.
 */
mx_status mx_gemm_splitk_noalloc(const mx_tensor* A, const mx_tensor* B, void* C,
                                 int32_t c_dtype, int64_t ldc, void* stream);

/* Synchronize the stream, then return (and clear) the first error recorded
 * by a kernel of this library on the current device: MX_OK,
 * MX_ERR_TIMEOUT, or MX_ERR_CUDA if the synchronization itself failed. */
mx_status mx_last_error(void* stream);

/* Failure-detection self test: launch one small kernel that waits, with a
 * bound of limit_cycles SM clock cycles (1 .. 2^40), on an mbarrier that
 * nothing ever arrives at.  The wait runs out, the kernel records
 * MX_ERR_TIMEOUT in the status word and returns; the context stays usable.
 * A following mx_last_error(stream) returns MX_ERR_TIMEOUT. */
mx_status mx_selftest_wait_timeout(int64_t limit_cycles, void* stream);

/* Host-only helper: convert a tiled scale plane (host memory,
 * mx_scale_bytes(outer, K) bytes) into the row-major outer x K/32 scale
 * matrix (host memory).  Not used on the GPU path. */
mx_status mx_scales_to_rowmajor(const uint8_t* tiled, uint8_t* rowmajor,
                                int64_t outer, int64_t K);

/* Name of a status code (static string). */
const char* mx_status_string(int32_t status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t mx_version(void);

/* Tuning and testing knob (the pages have no counterpart): the width of the
 * GEMMs' output tiles.  0 (the default) picks, per shape, the plan with the
 * smallest estimated time among 256-wide tiles, 128-wide tiles and -- for the
 * *_splitk calls -- 128-wide tiles with the K-split.  128 or 256 fixes the
 * width for every later mx_gemm / gemm_f16 call of the process (128 only
 * applies to fp32 / bf16 outputs: an MX-quantized C always uses 256).  The
 * K-split runs on 128-wide tiles: with 128 fixed, the *_splitk calls split
 * whenever the tiles leave part of a wave idle (and *_workspace_bytes sizes
 * the workspace for that); with 256 fixed they never split.
 * Results do not depend on the width (each element of C is summed in the
 * same order); they depend on the K-split only in the last bits.
 * Process-wide: set it while no other thread launches GEMMs.  Returns
 * MX_ERR_INVALID_ARG for any other value. */
mx_status mx_set_tile_width(int32_t tbn);

#ifdef __cplusplus
}
#endif

#endif /* MX_GB300_H */

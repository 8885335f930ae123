/*
 * mx.h -- C ABI of the GB300 (sm_103a) MX block-scaled quantization library.
 *
 * The library implements the hot path of OCP Microscaling (MX) block scaling:
 * quantize a float tensor into low-bit element codes plus one power-of-two
 * E8M0 scale per block of 32 consecutive elements along the last (reduction)
 * axis, dequantize it back exactly, and multiply two block-scaled operands
 * into an f32 accumulator that is both an input and the output.
 *
 * Sources (web pages, cited by title and section):
 *   [Dialect] "A Dialect Is a Set of Co-Designed Decisions: Designing for MX
 *             Quantization in MLIR" -- "The type: !mx.tensor", "The four ops",
 *             "The block axis", "The accumulator operand".
 *   [Layout]  "Bit Layout" (MXFP4 community format pages) -- "The E2M1
 *             element", "The E8M0 shared scale", "Block structure and
 *             packing", "Reference encode and decode".
 *
 * Conventions shared by every call
 *   - All tensor pointers are DEVICE pointers, owned by the caller.  The
 *     library allocates no device memory and keeps no pointer after a call
 *     returns.  Outputs are written in place (destination passing, [Dialect]
 *     "The accumulator operand").
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls are asynchronous on that stream.  Argument checks happen
 *     on the host before anything is launched; a failed check returns an error
 *     and launches nothing.
 *   - Tensors are row-major and dense.  A tensor of `rows` x `cols` is blocked
 *     along `cols`; `cols` must be a multiple of the block size 32 (the type
 *     verifier's rule: the block size divides the last dimension, [Dialect]
 *     "The type: !mx.tensor").  Zero rows or zero cols is a valid no-op.
 *   - block_size must be 32 and scale_type MX_SCALE_E8M0; anything else is
 *     MX_ERR_UNSUPPORTED.
 *   - Pointers must be 16-byte aligned (MX_ERR_ALIGN) unless stated.
 *   - There is no CPU fallback: without a usable CUDA device every compute
 *     call returns MX_ERR_CUDA or MX_ERR_NO_DEVICE.
 *
 * Element codes ([Layout] "The E2M1 element", "Block structure and packing")
 *   MX_E2M1   (MXFP4): 4-bit code S.EE.M, bias 1, magnitudes
 *             {0, .5, 1, 1.5, 2, 3, 4, 6}; two codes per byte, element 2k in
 *             the LOW nibble and element 2k+1 in the high nibble.  A row of
 *             `cols` elements is cols/2 bytes.
 *   MX_E4M3FN (MXFP8): 8-bit code S.EEEE.MMM, bias 7, largest finite 448,
 *             S.1111.111 is NaN, no infinities.  One byte per element.
 *
 * Scales ([Layout] "The E8M0 shared scale")
 *   One E8M0 byte b per block: value 2^(b-127); b = 0xFF is NaN and turns
 *   every element of its block into NaN.  Two layouts:
 *   MX_SCALES_ROWMAJOR: [rows][cols/32] bytes, row-major (the public layout).
 *   MX_SCALES_MMA: the tensor-core operand layout.  Rows are padded to a
 *     multiple of 128 and blocks per row to a multiple of 4; scale (r, j)
 *     (row r, block j) is the byte at
 *       ((r/128) * (NB4/4) + j/4) * 512 + (r%32)*16 + ((r/32)%4)*4 + (j%4)
 *     where NB4 = blocks per row rounded up to a multiple of 4.  Padding bytes
 *     are written as 0 by mx_quantize.  Size: mx_scales_bytes().
 *
 * Rounding ([Layout] "Reference encode and decode"; readings where the pages
 * are silent are marked *)
 *   amax = max |x| over the block; an all-zero block gets codes 0 and scale
 *   127.  e = floor(log2 amax) - emax (emax 2 for E2M1, 8* for E4M3FN), with
 *   floor(log2) the exact integer exponent*, clipped to [-127, 127]; scale
 *   byte e + 127.  Each element goes to the nearest grid magnitude of
 *   |x| / 2^e, ties to the LOWER magnitude*, saturating at the largest finite
 *   magnitude; the sign bit is set when x < 0.  A block holding a NaN or an
 *   infinity gets scale 0xFF and codes 0*.
 */
#ifndef MX_H
#define MX_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MX_API __attribute__((visibility("default")))
#else
#define MX_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MX_OK = 0,
    MX_ERR_NULL = 1,        /* a required pointer is NULL */
    MX_ERR_SHAPE = 2,       /* negative dimension, cols % 32 != 0, or a shape rule below */
    MX_ERR_UNSUPPORTED = 3, /* block_size != 32, scale type, format/dtype/layout value, aliasing */
    MX_ERR_ALIGN = 4,       /* pointer misaligned for the call */
    MX_ERR_TIMEOUT = 5,     /* a kernel gave up waiting (reported by mx_device_status) */
    MX_ERR_CUDA = 6,        /* a CUDA runtime or driver call failed */
    MX_ERR_NO_DEVICE = 7    /* no sm_103 device is current */
} mx_status_t;

typedef enum { MX_E2M1 = 1, MX_E4M3FN = 2 } mx_format_t;
typedef enum { MX_SCALE_E8M0 = 1 } mx_scale_type_t;
typedef enum { MX_F32 = 1, MX_BF16 = 2 } mx_dtype_t;
typedef enum { MX_SCALES_ROWMAJOR = 0, MX_SCALES_MMA = 1 } mx_scale_layout_t;

/* Bytes of element codes for a rows x cols tensor in format fmt
 * (rows*cols/2 for E2M1, rows*cols for E4M3FN); -1 on a bad argument. */
MX_API int64_t mx_codes_bytes(mx_format_t fmt, int64_t rows, int64_t cols);

/* Bytes of scales for a rows x cols tensor in the given scale layout
 * (rows*cols/32 row-major; the padded size for MX_SCALES_MMA); -1 on a bad
 * argument.  One scale per block: the count is a property of the type, not
 * of the data ([Dialect] "The type: !mx.tensor", getNumScaleBlocks). */
MX_API int64_t mx_scales_bytes(mx_scale_layout_t layout, int64_t rows, int64_t cols);

/* quantize_block over a whole tensor ([Dialect] "The four ops";
 * [Layout] "Reference encode and decode").
 *   x       : rows x cols input, f32 or bf16 (x_dtype), row-major, 16-B aligned.
 *   codes   : out, mx_codes_bytes(fmt, rows, cols) bytes, 16-B aligned.
 *   scales  : out, mx_scales_bytes(scale_layout, rows, cols) bytes; 4-B
 *             aligned for MX_SCALES_ROWMAJOR, 16-B for MX_SCALES_MMA.
 * Codes and scales are bit-exact functions of x (see "Rounding" above). */
MX_API mx_status_t mx_quantize(const void* x, mx_dtype_t x_dtype, int64_t rows, int64_t cols,
                        mx_format_t fmt, int block_size, mx_scale_type_t scale_type,
                        void* codes, uint8_t* scales, mx_scale_layout_t scale_layout,
                        void* stream);

/* dequantize_block over a whole tensor ([Dialect] "The four ops": back to
 * f32; [Layout] "The E8M0 shared scale").  y[r][c] = element * 2^(b-127),
 * exact (no rounding step); b = 0xFF gives NaN for the whole block, as does
 * an E4M3FN NaN code for its element.  Subnormal results are kept.
 *   codes, scales : as written by mx_quantize (same fmt and scale_layout).
 *   y             : out, rows x cols f32, row-major, 16-B aligned. */
MX_API mx_status_t mx_dequantize(const void* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                          mx_format_t fmt, int block_size, mx_scale_type_t scale_type,
                          mx_scale_layout_t scale_layout, float* y, void* stream);

/* block_matmul ([Dialect] "The four ops", "The block axis", "The accumulator
 * operand"): C <- C + A * B, multiplied while both operands are still block
 * scaled, accumulated in f32 on the tensor cores, C updated in place.
 *   A : M x K, codes a_codes (format a_fmt) and scales a_scales, blocked
 *       along K.
 *   B : K x N, passed TRANSPOSED as an N x K tensor (b_codes, b_scales,
 *       format b_fmt) so that it too is blocked along its reduction axis K
 *       ([Dialect] "The block axis": the law is reduction-axis blocking).
 *   scale_layout : layout of both a_scales and b_scales.  MX_SCALES_MMA is the
 *       fast path (one bulk copy per scale tile); MX_SCALES_ROWMAJOR is accepted
 *       when K % 128 == 0 (the kernel gathers 4-byte scale words itself).
 *   C : M x N f32, row-major, read and written in place; must not overlap an
 *       input (MX_ERR_UNSUPPORTED).
 * Formats: any pair of MX_E2M1 / MX_E4M3FN.  Shape rules: K % 32 == 0; when
 * exactly one operand is MX_E2M1, K % 128 == 0 and that operand's codes must
 * be 32-B aligned.
 * Result: C[m][n] + sum_k deqA[m][k] * deqB[n][k], summed in f32 (order
 * unspecified; the parity bound is 1e-5 * sum_k |deqA*deqB|).  A NaN scale
 * or NaN code reaches the outputs that use it.  f32 subnormal results may be
 * flushed to zero by the tensor-core and reduction hardware. */
MX_API mx_status_t mx_block_matmul(const void* a_codes, const uint8_t* a_scales, mx_format_t a_fmt,
                            const void* b_codes, const uint8_t* b_scales, mx_format_t b_fmt,
                            mx_scale_layout_t scale_layout, int block_size,
                            mx_scale_type_t scale_type, int64_t M, int64_t N, int64_t K,
                            float* C, void* stream);

/* block_matmul with a caller-owned device workspace ([Dialect] "The four ops",
 * "The block axis", "The accumulator operand"; the workspace, like every
 * buffer here, is the caller's: destination passing).  Arguments and result
 * as mx_block_matmul.  With MX_SCALES_MMA the workspace is unused (may be
 * NULL) and the call is mx_block_matmul.  With MX_SCALES_ROWMAJOR (K % 128 ==
 * 0) both operands' scales are first rewritten into the workspace in the
 * tensor-core layout -- A's at byte 0, B's at the next 256-byte boundary --
 * by one small kernel on `stream`, and the product then runs as with
 * MX_SCALES_MMA (the row-major path of mx_block_matmul gathers scale words
 * inside the GEMM and is slower for most shapes).  The exception is decode
 * shapes -- M <= 32 with N > M, and K a multiple of 256 (512 when both
 * operands are MX_E2M1) -- where the gather costs about what the bulk scale
 * copies do: those calls are mx_block_matmul with row-major scales and leave
 * the workspace untouched (it is still validated).  The workspace is only
 * written; its previous contents do not matter.
 *   workspace       : device pointer, 256-byte aligned (MX_ERR_ALIGN), not
 *                     overlapping C or an input (MX_ERR_UNSUPPORTED).
 *   workspace_bytes : at least mx_block_matmul_workspace_bytes(...)
 *                     (MX_ERR_SHAPE otherwise; MX_ERR_NULL for a NULL
 *                     workspace that row-major scales need).
 * Asynchronous on `stream`; the workspace must stay allocated until the call
 * has run, and two calls that share a workspace must be ordered. */
MX_API mx_status_t mx_block_matmul_ws(const void* a_codes, const uint8_t* a_scales, mx_format_t a_fmt,
                               const void* b_codes, const uint8_t* b_scales, mx_format_t b_fmt,
                               mx_scale_layout_t scale_layout, int block_size, mx_scale_type_t scale_type,
                               int64_t M, int64_t N, int64_t K, float* C, void* workspace,
                               int64_t workspace_bytes, void* stream);

/* Bytes of workspace mx_block_matmul_ws needs: 0 for MX_SCALES_MMA or an empty
 * product; for MX_SCALES_ROWMAJOR the tensor-core-layout scale bytes of A and
 * of B, each rounded up to 256.  -1 for an invalid layout or shape. */
MX_API int64_t mx_block_matmul_workspace_bytes(mx_scale_layout_t scale_layout, int64_t M, int64_t N, int64_t K);

/* mx_block_matmul_ws for callers that cannot allocate device memory.  The
 * pages have no counterpart: this is a deployment variant.  Callers in this
 * position include a host framework or plugin runtime that owns every device
 * buffer and hands a library only its inputs and outputs, a process held to a
 * device memory budget fixed at start-up, and latency-critical code where an
 * allocation, which may synchronize the device, is not acceptable.
 * Arguments and result are those of mx_block_matmul; the caller still passes
 * every input and C.  The scratch for the tensor-core-layout scales is one
 * file-scope device array of 16 MiB (16777216 bytes), which every GPU that
 * loads the library holds until the process exits, so products whose
 * mx_block_matmul_workspace_bytes exceed that are rejected with MX_ERR_SHAPE
 * (for example M = N = K = 8192 needs 4 MiB, M = 8192, N = 28672, K = 8192
 * needs 9 MiB).  The call allocates nothing: no cudaMalloc, cudaFree or other
 * allocating routine.
 * Every call shares that one array, which keeps the last call's contents; a
 * call rewrites every byte it reads, so nothing needs clearing, but calls that
 * overlap on the GPU (other streams, or host threads without ordering between
 * their calls) race on it and can produce wrong results.  The first call on a
 * device looks up the array's device address (set-up, once per device) and
 * should come before any stream capture.  With MX_SCALES_MMA no scratch is
 * used and the call is mx_block_matmul. */
MX_API mx_status_t mx_block_matmul_static_ws(const void* a_codes, const uint8_t* a_scales, mx_format_t a_fmt,
                                      const void* b_codes, const uint8_t* b_scales, mx_format_t b_fmt,
                                      mx_scale_layout_t scale_layout, int block_size,
                                      mx_scale_type_t scale_type, int64_t M, int64_t N, int64_t K, float* C,
                                      void* stream);

/* quantize_block along an explicit block axis ([Dialect] "The block axis":
 * blocks run along the reduction axis, which for the right-hand operand of a
 * product is its first axis).
 *   axis = 1 : exactly mx_quantize (blocks of 32 along cols; cols % 32 == 0).
 *   axis = 0 : blocks of 32 consecutive ROWS of one column (rows % 32 == 0,
 *              cols any).  Outputs are laid out as the transposed tensor's
 *              would be: codes mx_codes_bytes(fmt, cols, rows) bytes, row c
 *              holding column c's codes; scales mx_scales_bytes(scale_layout,
 *              cols, rows), with cols as the scale layout's rows.  The result
 *              is directly the N x K operand B of mx_block_matmul for a K x N
 *              input.  Codes and scales equal mx_quantize of the transpose.
 * Other arguments, alignment and errors as mx_quantize; axis outside {0, 1}
 * is MX_ERR_UNSUPPORTED. */
MX_API mx_status_t mx_quantize_axis(const void* x, mx_dtype_t x_dtype, int64_t rows, int64_t cols, int axis,
                             mx_format_t fmt, int block_size, mx_scale_type_t scale_type, void* codes,
                             uint8_t* scales, mx_scale_layout_t scale_layout, void* stream);

/* dequantize_block with a bfloat16 result ([Dialect] "The four ops").  Each
 * element is the exact value of mx_dequantize rounded to the nearest bfloat16,
 * ties to even; 0xFF scales and E4M3FN NaN codes give NaN.
 *   y : out, rows x cols bfloat16 (2 bytes each), row-major, 16-B aligned.
 * Other arguments and errors as mx_dequantize. */
MX_API mx_status_t mx_dequantize_bf16(const void* codes, const uint8_t* scales, int64_t rows, int64_t cols,
                               mx_format_t fmt, int block_size, mx_scale_type_t scale_type,
                               mx_scale_layout_t scale_layout, void* y, void* stream);

/* fold_scale ([Dialect] "The four ops"): multiply the MX tensor whose scales
 * these are (rows x cols elements) by `scalar`, in place, by adding j to every
 * scale byte where scalar = 2^j ([Layout] "The E8M0 shared scale": the byte is
 * the exponent of a power of two).  A byte saturates at 0 (2^-127) and 254
 * (2^127); 0xFF stays NaN; the codes are untouched; the padding of
 * MX_SCALES_MMA stays 0.  The result is exact wherever no byte saturates.
 * A scalar that is not a positive finite power of two cannot be folded:
 * MX_ERR_UNSUPPORTED, nothing launched. */
MX_API mx_status_t mx_fold_scale(uint8_t* scales, int64_t rows, int64_t cols, mx_scale_layout_t scale_layout,
                          double scalar, void* stream);

/* block_matmul with an unquantized right operand ([Dialect] "The four ops":
 * the first form of block_matmul, an MX tensor times a plain f32 one):
 *   C <- C + dequantize(A) * B
 *   A : M x K codes (a_fmt) with scales in a_scale_layout, blocked along K.
 *   B : K x N f32, row-major (not transposed, no scales).
 *   C : M x N f32, row-major, read and written in place.
 * Each output is the exact sum of C and the products deq(a)*b, up to f32
 * rounding: partial sums are formed per 32-element block of A and per share
 * of K, so |C - exact| stays within 1e-5 * sum |deq(a) * b|.  The order in
 * which the shares of K are added into C is not fixed, so repeated calls may
 * differ in the last bits.  A 0xFF scale poisons its block: every output
 * that uses the block is NaN.
 * N % 4 == 0 (rows of B and C start on 16-byte boundaries: MX_ERR_ALIGN
 * otherwise); all four pointers 16-B aligned; K % 32 == 0; C must not
 * overlap an input.  An empty product returns MX_OK without launching. */
MX_API mx_status_t mx_block_matmul_f32b(const void* a_codes, const uint8_t* a_scales, mx_format_t a_fmt,
                                 mx_scale_layout_t a_scale_layout, int block_size, mx_scale_type_t scale_type,
                                 const float* B, int64_t M, int64_t N, int64_t K, float* C, void* stream);

/* block_matmul with the activations quantized on the fly ([Dialect] "The
 * four ops": quantize_block then block_matmul, the step before the product
 * folded into it): C <- C + quantize(a) * B, where `a` is M x K f32 or bf16
 * (a_dtype), row-major, quantized to a_fmt along K exactly as mx_quantize
 * would (same codes, same scales), inside the GEMM kernel -- the quantized
 * activations never reach HBM.
 *   B : N x K codes (b_fmt) with scales in MX_SCALES_MMA (b_scale_layout must
 *       be MX_SCALES_MMA), as for mx_block_matmul.
 *   C : M x N f32, read and written in place.
 * For M <= 64 (decode-shaped products); a larger M returns MX_ERR_UNSUPPORTED
 * (quantize A once with mx_quantize and call mx_block_matmul: a larger A would
 * be quantized again for every column tile).  Formats: E4M3FN activations
 * with E4M3FN or E2M1 weights, E2M1 activations with E2M1 weights.  `a` must
 * be 32-B aligned; other rules, results and tolerance as mx_block_matmul.
 * Speed: bf16 activations with M <= 16 and K a multiple of 256 (E4M3FN
 * activations) or 512 (E2M1) match mx_quantize + mx_block_matmul in one
 * launch; f32 activations take about twice as long as those two calls. */
MX_API mx_status_t mx_block_matmul_act(const void* a, mx_dtype_t a_dtype, mx_format_t a_fmt, const void* b_codes,
                                const uint8_t* b_scales, mx_format_t b_fmt, mx_scale_layout_t b_scale_layout,
                                int block_size, mx_scale_type_t scale_type, int64_t M, int64_t N, int64_t K,
                                float* C, void* stream);

/* Re-lay scales between MX_SCALES_ROWMAJOR and MX_SCALES_MMA (both
 * directions; identical layouts copy).  src and dst must not overlap; sizes
 * as mx_scales_bytes().  The scale values are not changed. */
MX_API mx_status_t mx_scales_relayout(const uint8_t* src, mx_scale_layout_t src_layout, int64_t rows,
                               int64_t cols, uint8_t* dst, mx_scale_layout_t dst_layout,
                               void* stream);

/* Synchronize `stream`, then report and clear the device-side error word
 * that kernels set when a bounded wait gives up (MX_ERR_TIMEOUT), or the
 * stream's CUDA error (MX_ERR_CUDA).  MX_OK when neither happened.  After a
 * timeout the output of the launch that gave up is unspecified.  Before its
 * CTAs exit, the GEMM waits at least 1 s for the loads and MMAs it already
 * issued.  The one exception is the decode path of mx_block_matmul_act with
 * bf16 activations and M <= 16, whose wait after a give-up is bounded but
 * not certain to cover every load. */
MX_API mx_status_t mx_device_status(void* stream);

/* Failure-detection self test: launches one block that waits on a barrier
 * nothing will ever complete, giving up after `limit_ns` nanoseconds
 * (1e3..1e10); the kernel then sets the error word and returns normally, so
 * the context stays usable.  mx_device_status() afterwards must report
 * MX_ERR_TIMEOUT. */
MX_API mx_status_t mx_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Measurement helper, no counterpart in the method: the rate of the
 * block-scaled tensor-core MMA on this GPU, for the block_matmul roofline.
 * One CTA per SM issues `iters` x 4 MMAs of 128 x 256 x (32 E4M3FN or 64
 * E2M1) elements on operands resident in shared memory (fmt selects
 * kind::mxf8f6f4 with E4M3FN x E4M3FN, or kind::mxf4 with E2M1 x E2M1);
 * *tflops receives 2*M*N*K of all MMAs over the span from the first CTA's
 * start to the last CTA's end.  Synchronous (waits for `stream`).  iters in
 * 1..1000000 (MX_ERR_SHAPE otherwise); MX_ERR_TIMEOUT if a CTA's bounded wait
 * gave up.  The per-CTA times pass through one device array (at most 1024
 * CTAs) that every call shares: calls must not overlap, on any stream or host
 * thread.  Each CTA allocates all TMEM of its SM, so run it on an otherwise
 * idle GPU (the allocation waits while another kernel holds TMEM there). */
MX_API mx_status_t mx_measure_mma_rate(mx_format_t fmt, int iters, double* tflops, void* stream);

/* Static text for a status code. */
MX_API const char* mx_status_string(mx_status_t status);

/* Text describing the last error returned on the calling host thread
 * (empty string if none). */
MX_API const char* mx_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* MX_H */
